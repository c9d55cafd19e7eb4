"""Paged versus contiguous KV memory accounting (the block-size trade-off).

Pins: the pages' worked numbers (a 4,096-token reservation holding 287 tokens,
2,048 holding 200; 35 tokens in 16-token blocks -> 48 slots with 13 unused),
the fragmentation picture (a freed region between live ones too small for the
next request although enough memory is free in total), and invariants of the
simulation (block size 1 wastes nothing; paged waste stays below one block per
running request; every token is generated once when nothing is preempted).
The paged side runs on the library's own allocator, so the native library must
build (host code only; no GPU needed).
"""
import numpy as np
import pytest

from conftest import read_golden
from paged_kv_cache_276_gb300 import build, waste


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def test_page_reservation_examples():
    # x321.org "Why naive allocation wastes so much memory": 4,096 reserved, 287 used
    assert waste.contiguous_used_fraction(287, 4096) == pytest.approx(0.0700683, abs=1e-6)
    # praveentn.live "The situation": 2,048 reserved, 200 generated
    assert waste.contiguous_used_fraction(200, 2048) == pytest.approx(0.0976563, abs=1e-6)
    with pytest.raises(ValueError):
        waste.contiguous_used_fraction(300, 200)


def test_paged_slots_match_the_page_block_counts():
    for length, block, blocks, capacity, unused, _used_last, _o in read_golden("block_counts.txt"):
        assert waste.paged_slots(int(length), int(block)) == int(capacity)
        assert waste.paged_slots(int(length), int(block)) - int(length) == int(unused)


def test_first_fit_fragmentation_picture():
    ff = waste.FirstFit(350)
    a, b, c, d = ff.alloc(100), ff.alloc(100), ff.alloc(100), ff.alloc(50)
    assert (a, b, c, d) == (0, 100, 200, 300) and ff.total_free() == 0
    ff.release(b, 100)
    ff.release(d, 50)
    assert ff.total_free() == 150 and ff.largest_hole() == 100
    assert ff.alloc(120) is None  # enough memory in total, no hole large enough
    # blocks of 10: every free block fits every request
    res = waste.simulate([120], [121], 150, "paged", block_size=10)
    assert res.generated == 1 and res.peak_running == 1 and res.preemptions == 0
    ff.release(c, 100)  # coalesces with the hole left by b and d
    assert ff.free == [(100, 250)]


def _stream(n, seed, top=2000):
    rng = np.random.default_rng(seed)
    return waste.request_stream(rng.integers(1, top + 1, size=n), rng)


def test_block_size_one_wastes_nothing_and_waste_stays_below_a_block():
    p, f = _stream(40, 1)
    tr = []
    r1 = waste.simulate(p, f, 8 * 2000, "paged", block_size=1, trace=tr)
    assert r1.utilisation == 1.0 and all(h == pin for h, pin, _ in tr)
    for bs in (16, 64):
        tr = []
        r = waste.simulate(p, f, 8 * 2000, "paged", block_size=bs, trace=tr)
        assert all(0 <= pin - h < bs * max(1, run) for h, pin, run in tr)
        if r.preemptions == 0:
            assert r.generated == sum(fi - pi for pi, fi in zip(p, f))


def test_contiguous_reservation_pins_the_largest_request():
    p, f = _stream(30, 2)
    tr = []
    r = waste.simulate(p, f, 4 * 2000, "contiguous", reserve=2000, trace=tr)
    assert r.generated == sum(fi - pi for pi, fi in zip(p, f)) and r.preemptions == 0
    assert all(pin == 2000 * run for _, pin, run in tr)
    assert r.peak_running == 4  # four reservations fit
    with pytest.raises(ValueError):
        waste.simulate(p, f, 4 * 2000, "contiguous", reserve=100)


def test_paged_holds_more_token_state_than_contiguous_on_a_mixed_stream():
    p, f = _stream(60, 3, top=4096)
    cap = 8 * 4096
    c = waste.simulate(p, f, cap, "contiguous", reserve=4096)
    g = waste.simulate(p, f, cap, "paged", block_size=16)
    assert g.token_state_fraction > c.token_state_fraction
    assert g.mean_running > c.mean_running and g.steps < c.steps


def test_causal_visible_keys_matches_brute_force():
    from paged_kv_cache_276_gb300.workloads import causal_visible_keys
    rng = np.random.default_rng(3)
    for _ in range(200):
        B = int(rng.integers(1, 6))
        lens = rng.integers(0, 300, size=B)
        chunks = rng.integers(0, 320, size=B)
        brute = sum(max(0, int(L) - int(c) + 1 + r) for L, c in zip(lens, chunks) for r in range(int(c)))
        assert causal_visible_keys(lens, chunks) == brute
    # a whole prompt from an empty cache: c (c + 1) / 2
    assert causal_visible_keys([4096], [4096]) == 4096 * 4097 // 2
