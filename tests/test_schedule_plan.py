"""CPU checks of the whole-model CSA2 layer schedule (host logic only): the
layer counts and positions the pages print ("The 890-Byte Token", section
"CSA2 cross-layer KV and index reuse"; knowledge note, "CSA2: share cache,
refresh selection only when needed")."""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def S():
    # the schedule module is plain Python; load it without the CUDA library
    spec = importlib.util.spec_from_file_location(
        "csa2_schedule", os.path.join(ROOT, "fp4_kv_cache_rope_gb300", "schedule.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    return mod


def test_layer_counts_match_pages(S):
    plan = S.layer_plan()
    assert len(plan) == 38                                     # 40 layers minus 0 and 1
    full = [p.layer for p in plan if p.mode == S.FULL]
    reindex = [p.layer for p in plan if p.mode == S.REINDEX]
    reuse = [p.layer for p in plan if p.mode == S.REUSE]
    assert full == [2, 8, 14, 20]                              # cache-writing layers
    assert reindex == [24, 28, 32, 36]
    assert len(reuse) == 30
    assert sorted(full + reindex) == [2, 8, 14, 20, 24, 28, 32, 36]   # index-producing layers


def test_groups(S):
    plan = {p.layer: p for p in S.layer_plan()}
    for g, head in enumerate((2, 8, 14)):                      # encoder: Full + 5 Reuse, own cache
        for l in range(head, head + 6):
            assert plan[l].cache == g and plan[l].selection == head
    for head in (20, 24, 28, 32, 36):                          # decoder: one cache, groups of 4
        for l in range(head, head + 4):
            assert plan[l].cache == 3 and plan[l].selection == head
    assert all(plan[l].mode == S.REUSE for l in plan if l not in (2, 8, 14, 20, 24, 28, 32, 36))


@pytest.mark.parametrize("per_launch", [1, 2, 3, 4, 8])
def test_attention_chunks(S, per_launch):
    """Attention launches cover the 38 layers in order; a launch never mixes
    caches or selections and holds at most per_launch layers; the index call
    of a group precedes all of its launches (the group's head leads its first
    launch)."""
    plan = S.layer_plan()
    chunks = S.attention_chunks(plan, per_launch)
    assert [p for c in chunks for p in c] == plan
    for c in chunks:
        assert 1 <= len(c) <= per_launch
        assert len({(p.cache, p.selection) for p in c}) == 1
        assert all(p.mode == S.REUSE for p in c[1:])
    heads = [c[0].layer for c in chunks if c[0].mode != S.REUSE]
    assert heads == [2, 8, 14, 20, 24, 28, 32, 36]
    # fewest launches the groups allow: ceil(6 / n) per encoder group,
    # ceil(4 / n) per decoder group
    up = lambda a: -(-a // per_launch)
    assert len(chunks) == 3 * up(6) + 5 * up(4)
