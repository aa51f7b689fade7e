"""Pins for the reference block-utilisation simulation ("Serving" 23.4: the
96-block, 8-request demo; blocks handed out as a sequence grows waste less
than one block per sequence)."""
import random

from oracle.utilization import BS, blocks_for, demo_requests, simulate


def test_demo_reserving_the_maximum_runs_only_four():
    reqs = demo_requests()
    trace, admitted = simulate("reserve", 96, reqs, 700)
    assert max(s["running"] for s in trace) == 4
    assert any(a > r[0] for a, r in zip(admitted, reqs)), "later requests wait"
    assert all(s["blocks"] == 24 * s["running"] for s in trace)


def test_demo_paging_runs_every_request_on_arrival():
    reqs = demo_requests()
    trace, admitted = simulate("paged", 96, reqs, 700)
    assert admitted == [r[0] for r in reqs]
    assert max(s["running"] for s in trace) > 4
    assert max(s["blocks"] for s in trace) <= 96


def test_paged_waste_is_under_one_block_per_running_request():
    rnd = random.Random(3)
    reqs = [(rnd.randrange(200), rnd.randrange(1, 300), rnd.randrange(1, 300), 1024) for _ in range(40)]
    reqs.sort()
    trace, _ = simulate("paged", 4096, reqs, 900)
    for s in trace:
        assert 0 <= s["blocks"] * BS - s["tokens"] < BS * max(1, s["running"])
        assert s["blocks"] >= blocks_for(s["tokens"]) if s["running"] <= 1 else True


def test_tokens_held_are_prompt_plus_generated():
    reqs = [(0, 5, 3, 64), (1, 17, 2, 64)]
    trace, _ = simulate("paged", 16, reqs, 6)
    # step 0: request 0 holds 5 + 1; step 1: 5 + 2 and 17 + 1; step 2: 5 + 3 and 17 + 2;
    # request 0 finishes at the end of step 2, request 1 at the end of step 2 as well
    assert [s["tokens"] for s in trace[:3]] == [6, 25, 27]
    assert [s["running"] for s in trace[:4]] == [1, 2, 2, 0]
    assert [s["blocks"] for s in trace[:3]] == [1, 3, 3]


def test_reserve_needs_contiguous_space():
    # 4 blocks; request 0 takes blocks 0-1, request 1 blocks 2-3; after request 0
    # ends, a 3-block reservation cannot start until request 1 ends too
    reqs = [(0, 1, 2, 32), (0, 1, 6, 32), (1, 1, 1, 48)]
    trace, admitted = simulate("reserve", 4, reqs, 12)
    assert admitted[:2] == [0, 0] and admitted[2] == 6
