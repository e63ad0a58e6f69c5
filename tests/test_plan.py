"""Host-side planning through the C ABI (no GPU): the schedule rules of
mla_prolog_create and the longest-processing-time job assignment behind the
balanced job tables."""
import dataclasses
import itertools
import os
import random
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from mla_attention_prolog_gb300 import binding, workloads as wl  # noqa: E402

SMS = 152  # GB300


def cdiv(a, b):
    return (a + b - 1) // b


def job_bytes(T, NA, kb, bn, splits):
    """Operand bytes of each compression job in the kernel's job order (token
    tile, weight tile, K split): its K blocks x (token rows + weight rows) x
    128 bytes."""
    out = []
    for m in range(cdiv(T, 128)):
        for n in range(cdiv(NA, bn)):
            for sp in range(splits):
                nkb = (sp + 1) * kb // splits - sp * kb // splits
                rows = min(128, T - 128 * m)
                width = min(bn, NA - bn * n)
                out.append(nkb * 128 * (rows + width))
    return out


def greedy(cost, groups):
    """Independent restatement of the assignment rule: jobs by decreasing cost
    (ties by index), each to the least-loaded worker (lowest index on a tie)."""
    load = [0] * groups
    lists = [[] for _ in range(groups)]
    for j in sorted(range(len(cost)), key=lambda j: (-cost[j], j)):
        g = min(range(groups), key=lambda g: (load[g], g))
        load[g] += cost[j]
        lists[g].append(j)
    return lists, max(load) if cost else 0


@pytest.mark.parametrize("name,T,bn_a,splits", [
    ("v3_prefill", 0, 256, 1),        # measured fastest: 2173 vs 2441 us (128) on GB300
    ("v2lite_prefill", 0, 144, 1),    # 128 jobs on 152 SMs (192: 96 jobs; 128 and 256 need split-K)
    ("v3_prefill", 385, 128, 2),      # the wide tiles would need split-K 4 (measured slower)
    ("v3_decode", 0, 112, 8),         # 19 tiles x 8 splits = 152 CTAs
    ("v2lite_decode", 0, 112, 16),    # 6 tiles x 16 splits = 96 CTAs
])
def test_default_schedules(name, T, bn_a, splits):
    d = wl.WORKLOADS[name].dims
    d = d.with_T(T) if T else d
    p = binding.plan(d, SMS)
    assert (p["bn_a"], p["splits_a"]) == (bn_a, splits), p
    assert p["decode"] == (cdiv(d.T, 128) <= 2)
    assert p["group_a"] == 4


def _random_dims(rng):
    Lq = rng.choice([0, 0, 512, 1536])
    flags = wl.QUANT_Q if Lq else 0
    return wl.Dims(T=rng.choice([1, 7, 64, 128, 129, 300, 1024, 4096, 16384]), D=16 * rng.randint(16, 448),
                   q_lora_rank=Lq, kv_lora_rank=16 * rng.randint(4, 40), rope_dim=rng.choice([16, 32, 64]),
                   num_heads=rng.choice([1, 2, 16, 128]), nope_dim=rng.choice([32, 64, 128]),
                   v_dim=rng.choice([32, 128]), max_pos=4096, flags=flags)


def test_plan_invariants_over_random_dims():
    rng = random.Random(7)
    for _ in range(40):
        d = _random_dims(rng)
        for sms in (8, 132, SMS):
            p = binding.plan(d, sms)
            NA = d.q_lora_rank + d.kv_lora_rank + d.rope_dim
            kb = cdiv(d.D, 64)
            assert p["compress_jobs"] == cdiv(NA, p["bn_a"]) * cdiv(d.T, 128) * p["splits_a"], (d, p)
            assert p["bn_a"] % 16 == 0 and p["splits_a"] >= 1 and p["splits_a"] <= max(1, kb)
            cost = job_bytes(d.T, NA, kb, p["bn_a"], p["splits_a"])
            assert sum(cost) > 0
            _, want = greedy(cost, sms)
            assert p["busiest_bytes"] == want, (d, sms, p)
            assert p["busiest_bytes"] >= max(max(cost), -(-sum(cost) // sms))
            if p["decode"]:
                assert p["compress_jobs"] <= sms or p["splits_a"] == 1, (d, sms, p)
            else:
                assert p["bn_a"] in (128, 144, 192, 256)


def test_wide_default_needs_no_split():
    """A 144-, 192- or 256-wide default compression tile never comes with split-K."""
    rng = random.Random(11)
    for _ in range(60):
        d = dataclasses.replace(_random_dims(rng), T=rng.choice([512, 2048, 4096, 16384]))
        p = binding.plan(d, SMS)
        if p["bn_a"] > 128:
            assert p["splits_a"] == 1, (d, p)


def test_lpt_assigns_every_job_once_and_matches_the_rule():
    rng = random.Random(3)
    for _ in range(200):
        n = rng.randint(0, 60)
        groups = rng.randint(1, 20)
        cost = [rng.choice([0, 1, 5, 17, 100, rng.randint(0, 10 ** 6)]) for _ in range(n)]
        lists, busiest = binding.lpt(cost, groups)
        assert sorted(j for l in lists for j in l) == list(range(n))
        assert busiest == max((sum(cost[j] for j in l) for l in lists), default=0)
        want_lists, want = greedy(cost, groups)
        assert busiest == want and lists == want_lists
        if n:
            assert busiest <= sum(cost) / groups + max(cost)  # list-scheduling bound


def _opt(cost, groups):
    best = None
    for assign in itertools.product(range(groups), repeat=len(cost)):
        load = [0] * groups
        for j, g in enumerate(assign):
            load[g] += cost[j]
        best = max(load) if best is None else min(best, max(load))
    return best


def test_lpt_within_grahams_bound_of_the_optimum():
    """Longest-first list scheduling is within 4/3 - 1/(3m) of the optimum
    (Graham 1969); brute force on small instances."""
    rng = random.Random(5)
    for _ in range(60):
        n = rng.randint(1, 8)
        groups = rng.randint(1, 3)
        cost = [rng.randint(1, 50) for _ in range(n)]
        _, busiest = binding.lpt(cost, groups)
        opt = _opt(cost, groups)
        assert opt <= busiest <= (4 / 3 - 1 / (3 * groups)) * opt + 1e-9, (cost, groups, busiest, opt)


def test_plan_and_lpt_reject_bad_arguments():
    d = wl.WORKLOADS["tiny"].dims
    with pytest.raises(binding.MlaPrologError):
        binding.plan(d, 0)
    with pytest.raises(binding.MlaPrologError):
        binding.plan(dataclasses.replace(d, D=100), SMS)  # not a multiple of 16
    with pytest.raises(binding.MlaPrologError):
        binding.lpt([1, -2, 3], 2)
    with pytest.raises(binding.MlaPrologError):
        binding.lpt([1, 2], 0)
    assert binding.lpt([], 3) == ([[], [], []], 0)


def _constant(name):
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "mla_attention_prolog_gb300",
                            "csrc", "prolog.cuh")).read()
    return int(re.search(r"constexpr\s+\w+\s+%s\s*=\s*(\d+)\s*;" % name, src).group(1))


def test_w8a8_exact_chain_bounds():
    """The W8A8 integer products stay exact in FP32 accumulation: a chain of
    kW8ChainKb K blocks of 64 codes sums at most 64 kW8ChainKb 127^2 < 2^24
    in magnitude (one more block would pass it), and a row with
    sum |code| <= kW8SumLimit keeps every partial sum below 2^24 against
    weight codes of magnitude <= 127 (one more would not)."""
    kb, lim, bk = _constant("kW8ChainKb"), _constant("kW8SumLimit"), _constant("kBK")
    assert bk * kb * 127 ** 2 < 2 ** 24 <= bk * (kb + 1) * 127 ** 2
    assert lim * 127 < 2 ** 24 <= (lim + 1) * 127
    # a K of up to kW8ChainKb blocks never needs the mark: the largest possible sum |code| is within the limit
    assert bk * kb * 127 <= lim


@pytest.mark.parametrize("name,T,sms,want", [
    ("v2lite_prefill", 0, 152, 56),    # 512 jobs: 3 rounds + 56, which fit 112 CTAs as halves
    ("v2lite_prefill", 0, 148, 68),    # 512 = 3 x 148 + 68
    ("v2lite_prefill", 0, 132, 0),     # 512 = 3 x 132 + 116: 232 halves would not fit one round
    ("v2lite_prefill", 300, 152, 0),   # 48 jobs: one round
    ("v2lite_decode", 0, 152, 0),      # decode schedule
    ("v3_prefill", 0, 152, 0),         # a q path: the pair kernels (the kv-resident kernel plans its own)
])
def test_last_round_half_tiles(name, T, sms, want):
    """The KV-only prefill's last round of expansion jobs as half tiles: the
    remainder of the jobs over the CTAs when it fits twice into the grid."""
    w = wl.WORKLOADS[name]
    d = w.dims.with_T(T) if T else w.dims
    assert binding.plan(d, sms)["kv_halves"] == want
