"""The expert cache's host logic without a GPU (no slot table on the device,
a recording fetch): page spark_model/layers/moe_v41.rs module doc (the
ExpertLru: picked experts gathered into slots, misses read from the source)
and page .../moe_v41/device_route.rs (misses fetched, slot changes to the
table). Least recently used slots are reused first; hits are never evicted
by the request that touches them."""
import pytest

import moe_decode_quantized_gb300 as moe

ARENA = moe.Arena(base=1 << 30, slot_bytes=1 << 20, gate_off=0, up_off=1 << 16, down_off=1 << 17)


def _cache(n_slots, n_layers=2, n_routed=8):
    calls = []

    def fetch(layer, expert, addr, nbytes, stream):
        calls.append((layer, expert, (addr - ARENA.base) // ARENA.slot_bytes))
        assert nbytes == ARENA.slot_bytes
        return 0

    return moe.ExpertCache(n_layers, n_routed, n_slots, ARENA, None, fetch), calls


def test_misses_fill_free_slots_then_hits():
    c, calls = _cache(4)
    assert c.ensure(0, [3, 5, 3], stream=0) == 2          # repeats count once
    assert [x[:2] for x in calls] == [(0, 3), (0, 5)]
    assert len({x[2] for x in calls}) == 2      # two different slots
    assert c.ensure(0, [5, 3], stream=0) == 0             # both resident
    assert c.stats() == (2, 2, 0)
    assert c.slot_of(0, 3) == calls[0][2] and c.slot_of(0, 5) == calls[1][2]
    assert c.slot_of(1, 3) == -1                # layers are separate


def test_least_recently_used_slot_is_reused():
    c, calls = _cache(3)
    c.ensure(0, [0], stream=0)
    c.ensure(0, [1], stream=0)
    c.ensure(1, [2], stream=0)
    c.ensure(0, [0], stream=0)                            # 0 becomes most recently used
    s1 = c.slot_of(0, 1)
    assert c.ensure(1, [7], stream=0) == 1                # evicts (0, 1): the least recently used
    assert c.slot_of(0, 1) == -1 and c.slot_of(1, 7) == s1
    assert c.stats()[2] == 1
    assert calls[-1] == (1, 7, s1)


def test_a_request_never_evicts_its_own_hits():
    c, _ = _cache(3)
    c.ensure(0, [0, 1, 2], stream=0)
    # 0 and 1 are hits of this request; the one miss must take 2's slot
    s2 = c.slot_of(0, 2)
    assert c.ensure(0, [1, 0, 6], stream=0) == 1
    assert c.slot_of(0, 2) == -1 and c.slot_of(0, 6) == s2
    assert c.slot_of(0, 0) >= 0 and c.slot_of(0, 1) >= 0


def test_more_experts_than_slots_at_once_is_refused():
    c, _ = _cache(2)
    with pytest.raises(moe.MoeError) as e:
        c.ensure(0, [0, 1, 2], stream=0)
    assert e.value.code == -2
    with pytest.raises(moe.MoeError):
        c.ensure(0, [9], stream=0)                        # expert outside the layer
    with pytest.raises(moe.MoeError):
        c.ensure(5, [0], stream=0)                        # layer outside the cache


def test_a_failing_source_is_reported():
    c = moe.ExpertCache(1, 4, 2, ARENA, None, lambda l, e, a, b, s: 7)
    with pytest.raises(moe.MoeError) as e:
        c.ensure(0, [1], stream=0)
    assert e.value.code == -3 and "source failed" in str(e.value)
