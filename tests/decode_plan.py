"""The split-KV decode's documented plan, written out in Python for the tests.

The split kernel and the merge kernel compute the same plan on the device; the GPU tests
check the partials in the workspace against the key ranges this model gives, and the CPU
tests check the model's own invariants (every key of every (sequence, kv head) pair in
exactly one piece, consecutive slots, at most num_splits pieces per pair).
"""


def kv_group(Hkv, grid):
    """g: the kv heads planned as one entry (the largest of 8, 4 and 2 that divides Hkv
    and is at most the SM count, else 1)."""
    return next((c for c in (8, 4, 2) if Hkv % c == 0 and grid >= c), 1)


def pieces(lens, Hkv, ns, grid):
    """Key ranges of the split kernel's partials, as the API documents them: the 128-key
    tiles of all (sequence, kv head) pairs laid end to end in (b, kv head) order and cut
    into ranges of W tiles.  The kv heads are planned in groups of g adjacent heads
    (kv_group): a group's tiles count once, there is one range per g CTAs (the SM count
    rounded down to a multiple of g), and every head of a group gets the same pieces.
    W is the total over the ranges, but at least ceil(T / (ns - 1)) for the longest
    pair's T tiles (ns = 1: one range holds everything).  The head dim does not enter the
    plan.  Returns {(b, hk): [(slot, k0, k1), ...]}."""
    g = kv_group(Hkv, grid)
    ranges = (grid - grid % g) // g
    hu = Hkv // g
    tiles = [(n + 127) // 128 for n in lens]
    prefix = [0]
    for t in tiles:
        prefix.append(prefix[-1] + t)
    total = hu * prefix[-1]
    w = (total + ranges - 1) // ranges
    w = max(w, (max(tiles) + ns - 2) // (ns - 1)) if ns >= 2 else max(w, total)
    w = max(w, 1)
    out = {}
    for b, tb in enumerate(tiles):
        for hk in range(Hkv):
            start = hu * prefix[b] + (hk // g) * tb
            x, segs = start, []
            while x < start + tb:
                end = min((x // w + 1) * w, start + tb)
                segs.append((x // w - start // w, (x - start) * 128, min((end - start) * 128, lens[b])))
                x = end
            out[(b, hk)] = segs
    return out
