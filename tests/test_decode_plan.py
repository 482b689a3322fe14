"""CPU checks of the split-KV decode's plan model (tests/decode_plan.py), which the GPU
tests hold the kernels' partials to: over random length mixes, kv head counts, split
counts and SM counts, every key of every (sequence, kv head) pair lies in exactly one
piece, a pair's pieces take slots 0, 1, ... in key order and number at most num_splits,
and the heads of one planned group are cut identically.
"""
import random

from decode_plan import kv_group, pieces


def test_kv_group_rule():
    assert [kv_group(h, 152) for h in (1, 2, 3, 4, 6, 8, 12, 16, 32)] == [1, 2, 1, 4, 2, 8, 4, 8, 8]
    assert kv_group(8, 4) == 4 and kv_group(8, 1) == 1


def test_plan_covers_every_key_once():
    rng = random.Random(2024)
    for _ in range(1500):
        B = rng.randint(1, 24)
        Hkv = rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 32])
        ns = rng.choice([1, 2, 3, 5, 8, 19, 64])
        grid = rng.choice([1, 2, 3, 7, 8, 148, 152])
        lens = [rng.choice([0, 1, 127, 128, 129, rng.randint(0, 40000)]) for _ in range(B)]
        if max(lens) == 0:
            lens[0] = 1
        plan = pieces(lens, Hkv, ns, grid)
        g = kv_group(Hkv, grid)
        for b in range(B):
            for hk in range(Hkv):
                segs = plan[(b, hk)]
                assert [s for s, _, _ in segs] == list(range(len(segs)))
                assert len(segs) <= ns
                edge = 0
                for _, k0, k1 in segs:
                    assert k0 == edge and k1 > k0
                    edge = k1
                assert edge == lens[b]
                assert segs == plan[(b, hk - hk % g)]
