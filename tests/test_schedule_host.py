"""The tiled kernels' work split, checked on the host (no GPU needed).

`dspark_describe_schedule` returns the split the library plans
(csrc/internal.h, plan_schedule).  The walk each worker makes through it
(csrc/kernel_common.cuh: work_begin, work_next, sk_owner) is restated below
and driven over many problem shapes; the checks are the properties the
kernels rely on:

* every (tile, k-block) unit is computed exactly once;
* a worker publishes at most one part per workspace slot: slot 1 for a part
  that starts at the tile's first k-block, slot 0 otherwise, which is also
  how a reader finds a contributor's part (slot 1 iff it is the tile's first
  contributor);
* whole-tiles-first order: the owner of a cut tile's last k-block computes it
  as the last item of its walk (it finishes the tile), so waits only point to
  lower-numbered workers;
* split-first order: a worker's cut parts all come before its whole tiles,
  every worker ends on a whole tile, and the contributors' row shares of a cut
  tile partition its rows;
* one arrival counter per cut tile (indexed by the tile's last contributor).

The GPU parity tests cover the kernels that execute this walk.
"""
import pytest

import draft_model_kv_gb300 as dk
from draft_model_kv_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()   # host code only: nvcc builds here without a GPU


def walk(plan, wid, num_kb):
    """One worker's items (tile, kb0, kb1) in order (kernel_common.cuh)."""
    nw, dp, units, skw, first = (plan["workers"], plan["whole_tiles"], plan["split_units"],
                                 plan["split_workers"], plan["split_first"])
    start = cur = 0
    if wid < skw:
        start = wid * units // skw
        cur = (wid + 1) * units // skw
    dp_tile = wid
    items = []
    while True:
        if not first and dp_tile < dp:
            items.append((dp_tile, 0, num_kb))
            dp_tile += nw
            continue
        if cur > start:
            t = (cur - 1) // num_kb
            lo = max(start, t * num_kb)
            items.append((dp + t, lo - t * num_kb, cur - t * num_kb))
            cur = lo
            continue
        if first and dp_tile < dp:
            items.append((dp_tile, 0, num_kb))
            dp_tile += nw
            continue
        return items


def owner(plan, u):
    return ((u + 1) * plan["split_workers"] - 1) // plan["split_units"]


SHAPES = ([(t, kb, w) for t in (1, 2, 5, 31, 76, 77, 80, 94, 100, 101, 120, 151, 152, 160, 228, 230, 300)
           for kb in (1, 2, 3, 7, 64, 192) for w in (1, 3, 64, 76, 152)]
          + [(5120, 64, 76), (1024, 80, 76), (320, 112, 76), (40, 64, 152), (32, 192, 76)])


@pytest.mark.parametrize("allowed", [True, False])
def test_work_split_properties(allowed):
    for tiles, num_kb, workers in SHAPES:
        plan = dk.dspark_describe_schedule(tiles, num_kb, workers, allowed)
        nw = plan["workers"]
        assert 1 <= nw <= workers
        assert plan["whole_tiles"] + plan["split_units"] // num_kb == tiles
        assert plan["split_units"] % num_kb == 0
        if not allowed:
            assert plan["split_first"] == 0
        done = {}
        slots = set()
        for w in range(nw):
            items = walk(plan, w, num_kb)
            seen_whole = False
            for i, (tile, kb0, kb1) in enumerate(items):
                assert 0 <= tile < tiles and 0 <= kb0 < kb1 <= num_kb
                for k in range(kb0, kb1):
                    assert (tile, k) not in done, (tiles, num_kb, workers, tile, k)
                    done[(tile, k)] = w
                cut = kb0 != 0 or kb1 != num_kb
                if cut:
                    slot = 1 if kb0 == 0 else 0
                    assert (w, slot) not in slots
                    slots.add((w, slot))
                    u0 = (tile - plan["whole_tiles"]) * num_kb
                    if plan["split_first"]:
                        assert not seen_whole
                    elif owner(plan, u0 + num_kb - 1) == w:
                        assert i == len(items) - 1, "the finisher's piece is its last item"
                if tile < plan["whole_tiles"]:
                    seen_whole = True
            if plan["split_first"] and items:
                assert items[-1][0] < plan["whole_tiles"], "every worker ends on a whole tile"
        assert len(done) == tiles * num_kb
        counters = set()
        for st in range(plan["split_units"] // num_kb):
            u0 = st * num_kb
            cf, cl = owner(plan, u0), owner(plan, u0 + num_kb - 1)
            tile = plan["whole_tiles"] + st
            assert done[(tile, 0)] == cf and done[(tile, num_kb - 1)] == cl
            if cf == cl:
                continue
            assert cl not in counters
            counters.add(cl)
            for c in range(cf, cl + 1):
                assert (c, 1 if c == cf else 0) in slots
            if plan["split_first"]:
                n = cl - cf + 1
                for rv in (1, 7, 104, 128):
                    rows = [r for i in range(n) for r in range(i * rv // n, (i + 1) * rv // n)]
                    assert rows == list(range(rv))


def test_decode_shapes_take_the_split_first_order():
    # 80 pair tiles of the 512-token decode write on 76 pairs: 4 leftover tiles
    p = dk.dspark_describe_schedule(80, 64, 76)
    assert p == {"workers": 76, "whole_tiles": 76, "split_units": 256, "split_workers": 76, "split_first": 1}
    # more than a third of a wave left over, or two waves: whole tiles first
    assert dk.dspark_describe_schedule(120, 64, 76)["split_first"] == 0
    p = dk.dspark_describe_schedule(5120, 64, 76)
    assert p["split_first"] == 0 and p["whole_tiles"] == 66 * 76
    # fewer tiles than workers: every k-block split, at least 8 per worker
    p = dk.dspark_describe_schedule(2, 3, 152)
    assert p["whole_tiles"] == 0 and p["workers"] == 1


def test_whole_tiles_when_at_least_half_as_many_tiles_as_workers():
    """The tiled write gives every tile whole to one worker (no cut tile, the
    other workers idle) when there are fewer tiles than workers but at least
    half as many; below half, and for the weight-streaming kernel
    (split_first_allowed 0, which needs every SM streaming), the tiles are cut
    over the workers as before."""
    for workers in (64, 76, 152):
        for tiles in range(1, workers):
            p = dk.dspark_describe_schedule(tiles, 64, workers, True)
            whole = 2 * tiles >= workers
            if whole:
                assert p == {"workers": tiles, "whole_tiles": tiles, "split_units": 0, "split_workers": 0,
                             "split_first": 0}, (tiles, workers, p)
            else:
                assert p["whole_tiles"] == 0 and p["split_units"] == tiles * 64, (tiles, workers, p)
            q = dk.dspark_describe_schedule(tiles, 64, workers, False)
            assert q["whole_tiles"] == 0 and q["split_units"] == tiles * 64, (tiles, workers, q)
    # 256 tokens on 76 CTA pairs: 40 tiles whole on 40 pairs; 20 (k3gqa) cut
    assert dk.dspark_describe_schedule(40, 64, 76)["workers"] == 40
    assert dk.dspark_describe_schedule(20, 112, 76)["whole_tiles"] == 0


def test_refusals():
    with pytest.raises(dk.DSparkError):
        dk.dspark_describe_schedule(0, 64, 76)
    with pytest.raises(dk.DSparkError):
        dk.dspark_describe_schedule(80, 0, 76)
    with pytest.raises(dk.DSparkError):
        dk.dspark_describe_schedule(80, 64, 0)
