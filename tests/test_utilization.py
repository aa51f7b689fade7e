"""The library's utilisation replay against the reference simulation, step by
step, on the 96-block demo and on synthetic lognormal request streams (host
code: runs without a GPU)."""
import random

import numpy as np
import pytest

from oracle.utilization import demo_requests, simulate


@pytest.fixture(scope="module")
def util():
    from paged_kv_cache_227_gb300 import utilization
    return utilization


def same(trace, ref_trace):
    assert [(s.step, s.running, s.blocks, s.tokens, s.admitted) for s in trace] == \
        [(s["step"], s["running"], s["blocks"], s["tokens"], s["admitted"]) for s in ref_trace]


def test_demo_schedule_is_the_references(util):
    assert [(r.arrival, r.prompt, r.output, r.max_tokens) for r in util.demo_requests()] == demo_requests()


@pytest.mark.parametrize("policy", ["reserve", "paged"])
def test_demo_matches_reference(util, policy):
    reqs = demo_requests()
    trace, adm = util.run(policy, 96, reqs, 700)
    ref_trace, ref_adm = simulate(policy, 96, reqs, 700)
    same(trace, ref_trace)
    assert adm == ref_adm


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lognormal_streams_match_reference(util, seed):
    # synthetic stand-ins for chat-request lengths: lognormal prompts and outputs
    rng = np.random.default_rng(seed)
    n = 60
    arr = np.sort(rng.integers(0, 400, n))
    pr = np.clip(np.round(np.exp(np.log(150) + 0.9 * rng.standard_normal(n))), 1, 2000).astype(int)
    outp = np.clip(np.round(np.exp(np.log(200) + 0.8 * rng.standard_normal(n))), 1, 2000).astype(int)
    reqs = [(int(a), int(p), int(o), 2048) for a, p, o in zip(arr, pr, outp)]
    for policy in ("reserve", "paged"):
        trace, adm = util.run(policy, 1024, reqs, 1500)
        ref_trace, ref_adm = simulate(policy, 1024, reqs, 1500)
        same(trace, ref_trace)
        assert adm == ref_adm
    paged, _ = util.run("paged", 1024, reqs, 1500)
    reserve, _ = util.run("reserve", 1024, reqs, 1500)
    assert util.utilisation(paged) > 0.9 > util.utilisation(reserve)
