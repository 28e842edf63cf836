"""Host logic of the host-streaming forward: the segment plan covers the sequence exactly, ramps up
and down by doubling, and keeps every segment but at most one a whole number of chunks."""
import pytest

from gated_deltanet_mixer_gdn2_gb300.host_stream import segment_plan


@pytest.mark.parametrize("T", [0, 1, 63, 64, 100, 1000, 4096, 5000, 32768, 70000])
@pytest.mark.parametrize("seg", [64, 192, 1024, 4096])
def test_plan_covers_sequence(T, seg):
    plan = segment_plan(T, seg, 64)
    assert sum(plan) == T
    assert all(n > 0 for n in plan)
    assert max(plan, default=0) <= max(64, seg // 64 * 64) or len(plan) == 1
    assert sum(n % 64 != 0 for n in plan) <= 1


def test_plan_ramps():
    plan = segment_plan(32768, 4096, 64)
    assert plan[:3] == [512, 1024, 2048] and plan[-3:] == [2048, 1024, 512]
    assert plan[3:-3].count(4096) == 6
