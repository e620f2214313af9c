"""Host logic of the double-buffered activation reload (no GPU): the reload
schedule never overwrites a buffer that a pending backward still reads, and the
VRAM guardrail falls back to one buffer."""
import pytest

from moe_expert_dispatch_stable_gb300.offload import choose_buffers, reload_schedule


@pytest.mark.parametrize("L", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 2])
def test_reload_schedule_is_safe_and_overlapped(L, n):
    plan = reload_schedule(L, n)
    assert [s.layer for s in plan] == list(range(L - 1, -1, -1))
    # simulate: buffer -> layer it holds; a reload into buffer b may only happen after
    # the backward of the layer that used b before
    done = set()
    holder = {}
    for i, s in enumerate(plan):
        if s.buffer in holder:
            prev = holder[s.buffer]
            assert s.after == prev, "must wait for the previous user of the buffer"
        else:
            assert s.after == -1
        holder[s.buffer] = s.layer
        done.add(s.layer)
        # with two buffers, reload i+1 does not depend on backward i (they overlap)
        if n == 2 and i + 1 < L:
            assert plan[i + 1].after != s.layer
    assert done == set(range(L))


def test_guardrail_picks_two_one_or_fails():
    GB = 1 << 30
    assert choose_buffers(4 * GB, 20 * GB, 2 * GB) == 2
    assert choose_buffers(4 * GB, 9 * GB, 2 * GB) == 1           # second buffer would eat the reserve
    assert choose_buffers(4 * GB, 20 * GB, 2 * GB, want=1) == 1
    with pytest.raises(MemoryError):
        choose_buffers(4 * GB, 3 * GB, 0)
    with pytest.raises(ValueError):
        reload_schedule(0, 2)
