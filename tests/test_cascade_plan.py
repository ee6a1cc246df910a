"""Host-side cascade grouping (pkv_cascade_plan, no GPU): the items it forms
obey the contract of cascade attention [mlxcel manual "KV Cache", §"Paged Decode
Storage and Kernels": groups sharing a whole-page prefix, gated by a minimum
member count and a minimum number of shared pages], checked by brute force on
seeded tables with a tree of shared prefixes."""
import random

import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()


def _whole(ctx, mb):
    return min(max(ctx, 0) // 16, mb)


def _check_items(bt, ctx, members, blocks, width, min_members, min_shared):
    seen = set()
    for i in range(members.shape[0]):
        mem = [int(x) for x in members[i] if x >= 0]
        assert max(min_members, 2) <= len(mem) <= width
        assert all(x < 0 for x in members[i][len(mem):]), "padding only at the end"
        nb = int(blocks[i])
        assert nb >= min_shared
        for m in mem:
            assert m not in seen, "a sequence in two items"
            seen.add(m)
            assert _whole(int(ctx[m]), bt.shape[1]) >= nb
            assert torch.equal(bt[m, :nb], bt[mem[0], :nb])
        # the item's shared prefix is the whole common prefix of its members
        if nb < min(_whole(int(ctx[m]), bt.shape[1]) for m in mem):
            assert not all(bt[m, nb] == bt[mem[0], nb] for m in mem)
    return seen


def _tree_tables(seed, n, mb):
    """Sequences that branch off a few shared stems at random depths."""
    rng = random.Random(seed)
    next_block = [0]

    def fresh(k):
        out = list(range(next_block[0], next_block[0] + k))
        next_block[0] += k
        return out
    stems = [fresh(mb) for _ in range(3)]
    bt = torch.full((n, mb), -1, dtype=torch.int32)
    ctx = torch.zeros(n, dtype=torch.int32)
    for s in range(n):
        c = rng.randint(0, mb * 16)
        nb = -(-c // 16)
        if rng.random() < 0.8:
            stem = stems[rng.randrange(3)]
            depth = rng.choice([0, 2, 5, 9, mb])
            row = stem[:min(depth, nb)] + fresh(max(nb - depth, 0))
        else:
            row = fresh(nb)
        bt[s, :nb] = torch.tensor(row[:nb], dtype=torch.int32)
        ctx[s] = c
    return bt, ctx


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("width,min_members,min_shared", [(4, 2, 1), (16, 3, 4), (2, 2, 2), (8, 5, 9)])
def test_plan_contract(seed, width, min_members, min_shared):
    bt, ctx = _tree_tables(seed, 60, 12)
    members, blocks = ops.pkv_cascade_plan(bt, ctx, width, min_members, min_shared)
    _check_items(bt, ctx, members, blocks, width, min_members, min_shared)


def test_plan_finds_constructed_groups():
    groups = [list(range(0, 9)), [9, 10, 11], [12, 13]]
    ctx = [100 + 16 * i for i in range(16)]
    w = W.build(name="t", seed=3, context_lens=ctx, num_heads=4, num_kv_heads=2, head_dim=64, cache="f16",
                prefix_groups=groups, shared_blocks=6)
    members, blocks = ops.pkv_cascade_plan(w.block_tables, w.context_lens, 4, 2, 4)
    _check_items(w.block_tables, w.context_lens, members, blocks, 4, 2, 4)
    got = sorted(sorted(int(x) for x in r if x >= 0) for r in members)
    cover = sorted(x for r in got for x in r)
    assert cover == list(range(14)), "every member of every group is placed"
    assert sorted(len(r) for r in got) == [2, 3, 3, 3, 3]   # 9 -> 3 + 3 + 3, 3, 2
    assert (blocks == 6).all()


def test_plan_thresholds():
    groups = [[0, 1, 2]]
    w = W.build(name="t", seed=4, context_lens=[200, 210, 220, 230], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="f16", prefix_groups=groups, shared_blocks=6)
    for mm, ms, n in ((2, 6, 1), (3, 6, 1), (4, 6, 0), (2, 7, 0)):
        members, _ = ops.pkv_cascade_plan(w.block_tables, w.context_lens, 4, mm, ms)
        assert members.shape[0] == n, (mm, ms)


def test_plan_partial_last_block_is_not_shared():
    # two sequences with identical tables but 40 tokens: only 2 whole pages
    bt = torch.tensor([[5, 6, 7, -1], [5, 6, 7, -1]], dtype=torch.int32)
    ctx = torch.tensor([40, 40], dtype=torch.int32)
    members, blocks = ops.pkv_cascade_plan(bt, ctx, 4, 2, 1)
    assert members.shape[0] == 1 and int(blocks[0]) == 2
    members, _ = ops.pkv_cascade_plan(bt, ctx, 4, 2, 3)
    assert members.shape[0] == 0


def test_plan_rejects_bad_arguments():
    bt = torch.zeros((2, 4), dtype=torch.int32)
    ctx = torch.tensor([64, 64], dtype=torch.int32)
    with pytest.raises(ops.PkvError):
        ops.pkv_cascade_plan(bt, ctx, 0)
    with pytest.raises(ops.PkvError):
        ops.pkv_cascade_plan(bt, ctx, 17)
