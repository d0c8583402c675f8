"""Host-side tests of the C ABI: no GPU, no compute calls.

The library loads and exports every symbol the header declares; the binning
rule matches the page's (runtime.dep page, _bins: the smallest key >= B, else
the largest key); plan tables, validation and serialisation behave as the
header documents.
"""
import os
import re

import numpy as np
import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "dep_projection.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dep_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(dep):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(dep.lib(), name), name
    assert sorted(dep.EXPORTS) == names


def bins_rule(keys, B):
    """The page's rule, restated: smallest key >= B, else the largest key."""
    at_least = [k for k in keys if k >= B]
    return min(at_least) if at_least else max(keys)


def test_bins_rule_matches_page(dep):
    rng = np.random.default_rng(0)
    for _ in range(500):
        keys = list(rng.choice(np.arange(1, 300), rng.integers(1, 10), replace=False))
        for B in list(rng.integers(1, 400, 10)) + [1, max(keys), max(keys) + 1]:
            i = dep.dep_bins_index(keys, int(B))
            assert keys[i] == bins_rule(keys, int(B))
    assert dep.dep_bins_index([], 3) == -1


def test_default_table_follows_split_rule(dep):
    """Default table: one entry per requested batch, split-K kinds for small
    batches (runtime.hybrid page, HybridAttention.__init__)."""
    plan = dep.dep_projection_plan_host(7168, 12288, [16, 1, 4, 2, 8, 4], 152)
    try:
        table = dep.dep_projection_plan_table(plan)
        assert [t.max_rows for t in table] == [1, 2, 4, 8, 16]
        for t in table:
            assert t.stages >= 2
            if t.max_rows <= 2:  # the smallest batches: warp split-K over whole rows
                assert t.kind == dep.DEP_KIND_ROWS and t.ctas >= 152
            elif t.max_rows <= 4:  # long rows, 112 tiles of 64 rows on 152 SMs: one tile per block, one piece
                assert (t.kind, t.tile_n, t.splits, t.cols) == (dep.DEP_KIND_TC_SPLIT, 64, 1, 16)
            else:  # 448 tiles of 16 rows, about 3 per SM: warp-level MMAs, no tensor memory
                assert (t.kind, t.tile_n, t.tile_k, t.stages, t.cols) == (dep.DEP_KIND_WARP_MMA, 16, 256, 4, 16)
        for B, key in [(1, 1), (3, 4), (5, 8), (16, 16), (17, 16), (1000, 16)]:
            assert dep.dep_projection_plan_query(plan, B).max_rows == key
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("N,K,rows,expect", [
    (7168, 12288, 16, True), (7168, 1536, 8, True), (7280, 7168, 16, True),   # 448-455 tiles of 16 rows
    (7168, 12288, 4, False),                                                   # too few rows
    (3640, 7168, 16, False), (14560, 7168, 16, False),                         # 228 / 910 tiles
])
def test_default_rule_warp_mma(dep, N, K, rows, expect):
    """The warp-level MMA kind (DEP_KIND_WARP_MMA) is the default for 6-16 rows
    where tiles of 16 weight rows number 2.5 to 4 per SM, with 3 stages of 256
    columns at K <= 2048 and 4 above."""
    plan = dep.dep_projection_plan_host(N, K, [rows], 152)
    try:
        t = dep.dep_projection_plan_query(plan, rows)
        assert (t.kind == dep.DEP_KIND_WARP_MMA) == expect, t
        if expect:
            assert (t.tile_n, t.cols, t.tile_k, t.stages) == (16, 16, 256, 3 if K <= 2048 else 4)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("N,K", [(14560, 7168), (7168, 12288), (49376, 7168), (333, 40000), (333, 60000)])
def test_default_rule_whole_rows(dep, N, K):
    """One and two x rows take the whole-row kind on 16-row tiles and stages of
    1024 columns: six stages at one row where they fit beside x in shared memory
    (else four), four at two rows; where x does not fit at all, another kind."""
    plan = dep.dep_projection_plan_host(N, K, [1, 2], 152)
    try:
        t1, t2 = (dep.dep_projection_plan_query(plan, B) for B in (1, 2))
        ring = 16 * 1024 * 2  # bytes of one stage
        for t, rows, want in ((t1, 1, 6), (t2, 2, 4)):
            x_bytes = rows * K * 2
            if x_bytes + 4 * ring > 227 * 1024:
                assert t.kind != dep.DEP_KIND_ROWS, t  # x and four stages do not fit
                continue
            assert (t.kind, t.tile_n, t.tile_k, t.cols) == (dep.DEP_KIND_ROWS, 16, 1024, rows), t
            fits6 = x_bytes + 6 * ring + 4096 <= 227 * 1024  # with room for barriers and alignment
            assert t.stages == (want if want == 4 or fits6 else 4), t
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_default_many_tiles_take_three_pieces(dep):
    plan = dep.dep_projection_plan_host(49376, 7168, [1, 4, 16, 32], 152)
    try:
        kinds = {t.max_rows: (t.kind, t.splits) for t in dep.dep_projection_plan_table(plan)}
        assert kinds[1] == (dep.DEP_KIND_ROWS, 0)
        assert kinds[4] == kinds[16] == (dep.DEP_KIND_TC_SPLIT, 3)  # 386 tiles > 152 SMs
        assert kinds[32] == (dep.DEP_KIND_TC_XM, 0)  # x on the MMA's M side, tiles of 112 rows
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_default_batches_when_none_given(dep):
    plan = dep.dep_projection_plan_host(14560, 7168, [], 152)
    try:
        table = dep.dep_projection_plan_table(plan)
        assert [t.max_rows for t in table] == [1, 2, 4, 8, 16, 32, 64, 128, 256]
        # 114 tiles of 128 rows nearly fill 152 SMs: whole tiles, one per block
        assert all((t.kind, t.splits) == (dep.DEP_KIND_TC_SPLIT, 1) for t in table if 2 < t.max_rows <= 16)
        # 32 to 128 rows: x on the MMA's M side against 152 tiles of 96 weight rows
        xm = [t for t in table if 32 <= t.max_rows <= 128]
        assert all((t.kind, t.tile_n, t.cols, t.ctas, t.splits) == (dep.DEP_KIND_TC_XM, 96, 128, 152, 0)
                   for t in xm)
        # 256 rows: pairs of CTAs (each half of K) on 76 tiles of 192 rows, 152 CTAs
        t = table[-1]
        assert (t.max_rows, t.kind, t.tile_n, t.cols, t.splits, t.ctas) == (256, dep.DEP_KIND_TC_XM, 192, 256, 2, 152)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("N,sms,whole,pairs,cluster", [
    (7168, 152, {64: 48}, {128: (96, 128, 150)}, {256: (256, 4, 112)}),  # o_proj: clusters at 256 rows
    (14560, 152, {64: 96, 128: 96}, {256: (192, 256, 152)}, {}),           # DSA: 152 tiles of 96 rows
    (49376, 152, {64: 112, 128: 112}, {256: (224, 256, 152)}, {}),         # KDA: 441 tiles, three waves
    (1000, 8, {64: 128, 128: 128}, {256: (256, 256, 8)}, {}),              # 8 tiles of 128 rows on 8 SMs
])
def test_default_rule_wide_batches(dep, N, sms, whole, pairs, cluster):
    """The default rule for 64-256 rows: x on the MMA's M side wherever x's
    bytes per 64-column step are at most 1.5x the weight's -- whole K per block
    on tiles of R rows (the smallest multiple of 16 that fills the SMs in as few
    waves as tiles of at most 128 rows allow), else pairs of blocks (a cluster
    of two, each half of K) on tiles of up to twice that (multiples of 32 up to
    256); otherwise a cluster of k = SMs / groups (at most 4) CTAs per group of
    two 128-row tiles."""
    plan = dep.dep_projection_plan_host(N, 7168, [64, 128, 256], sms)
    try:
        table = {t.max_rows: t for t in dep.dep_projection_plan_table(plan)}
        for b, R in whole.items():
            t = table[b]
            assert (t.kind, t.tile_n, t.cols, t.ctas, t.splits) == (dep.DEP_KIND_TC_XM, R, 128, sms, 0), (b, t)
            assert 2 * (64 if b <= 64 else 128) <= 3 * R
        for b, (R, cols, ctas) in pairs.items():
            t = table[b]
            assert (t.kind, t.tile_n, t.cols, t.ctas, t.splits) == (dep.DEP_KIND_TC_XM, R, cols, ctas, 2), (b, t)
            assert R % 32 == 0 and 2 * (b if b > 64 else 64) <= 3 * R
        for b, (rows, k, ctas) in cluster.items():
            t = table[b]
            assert (t.kind, t.tile_n, t.splits, t.ctas) == (dep.DEP_KIND_TC_CLUSTER, rows, k, ctas), (b, t)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("N,K,batches,sms,status", [
    (0, 64, [1], 152, "DEP_ERR_INVALID_ARG"),
    (64, 0, [1], 152, "DEP_ERR_INVALID_ARG"),
    (64, 12, [1], 152, "DEP_ERR_MISALIGNED"),
    (64, 100, [1], 152, "DEP_ERR_MISALIGNED"),
    (64, 64, [0], 152, "DEP_ERR_INVALID_ARG"),
    (64, 64, [-3], 152, "DEP_ERR_INVALID_ARG"),
    (64, 64, [1], 0, "DEP_ERR_INVALID_ARG"),
])
def test_plan_argument_errors(dep, N, K, batches, sms, status):
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_plan_host(N, K, batches, sms)
    assert e.value.status == getattr(dep, status)


def test_host_plan_cannot_run(dep):
    plan = dep.dep_projection_plan_host(64, 64, [1], 152)
    try:
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_run(plan, 16, 16, 16, 1, 0)
        assert e.value.status == dep.DEP_ERR_UNSUPPORTED
        with pytest.raises(dep.DepError) as e:
            dep.dep_projection_run(plan, 16, 16, 16, -1, 0)
        assert e.value.status == dep.DEP_ERR_INVALID_ARG
        # inspection and host-buffer entry points refuse a host-only plan before any CUDA call
        for call in (lambda: dep.dep_projection_plan_partials(plan, 4),
                     lambda: dep.dep_projection_plan_exchange(plan, 4),
                     lambda: dep.dep_projection_device_status(plan, 0),
                     lambda: dep.dep_projection_run_host(plan, 16, 16, 16, 1, 0)):
            with pytest.raises(dep.DepError) as e:
                call()
            assert e.value.status == dep.DEP_ERR_UNSUPPORTED
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_plan_set_validates_and_inserts(dep):
    plan = dep.dep_projection_plan_host(7168, 12288, [1, 16], 152)
    try:
        t = dep.dep_tactic_t(max_rows=3, kind=dep.DEP_KIND_SPLITK_FMA, ctas=152, tile_n=64, tile_k=256,
                             stages=3, cols=4)
        dep.dep_projection_plan_set(plan, t)
        assert [x.max_rows for x in dep.dep_projection_plan_table(plan)] == [1, 3, 16]
        assert dep.dep_projection_plan_query(plan, 2).cols == 4
        bad = dep.dep_tactic_t(**{**t.as_dict(), "cols": 3})
        with pytest.raises(dep.DepError):
            dep.dep_projection_plan_set(plan, bad)
        bad = dep.dep_tactic_t(**{**t.as_dict(), "kind": 9})
        with pytest.raises(dep.DepError):
            dep.dep_projection_plan_set(plan, bad)
        bad = dep.dep_tactic_t(**{**t.as_dict(), "stages": 40})
        with pytest.raises(dep.DepError):
            dep.dep_projection_plan_set(plan, bad)
    finally:
        dep.dep_projection_plan_destroy(plan)


@pytest.mark.parametrize("fields,ok", [
    ({}, True),                                            # 96-row tiles, one block of rows, 4 stages of 2 slices
    ({"tile_n": 104}, False),                              # MMA N must be a multiple of 16
    ({"tile_n": 272}, False),                              # ... up to 256
    ({"cols": 192}, False),                                # one or two blocks of 128 rows
    ({"tile_k": 192}, False),                              # 1, 2 or 4 slices per stage
    ({"stages": 5}, False),                                # 5 x 56 KB does not fit in shared memory
    ({"splits": 1}, True),                                 # 1 = whole K, as 0
    ({"splits": 3}, False),                                # pairs only
    ({"splits": 2}, True),                                 # pairs of blocks on 96-row tiles
    ({"splits": 2, "tile_n": 80}, False),                  # pairs need a multiple of 32
    ({"splits": 2, "ctas": 1}, False),                     # ... and at least one pair
    ({"splits": 2, "cols": 256, "tile_n": 192, "tile_k": 64, "stages": 4}, True),  # DSA at 256 rows
    ({"splits": 2, "cols": 256, "tile_n": 256, "tile_k": 64, "stages": 2}, False),  # partials > the ring
])
def test_x_on_m_tactic_validation(dep, fields, ok):
    """The x-on-M kind's tactic fields (DEP_KIND_TC_XM): MMA N (tile_n), blocks
    of batch rows per pass (cols), slices per stage (tile_k), ring depth that
    fits beside x at 128 rows, and pairs (splits = 2), whose ring must also hold
    the other block's partials."""
    plan = dep.dep_projection_plan_host(14560, 7168, [128], 152)
    try:
        t = dep.dep_tactic_t(**{**dict(max_rows=100, kind=dep.DEP_KIND_TC_XM, ctas=152, tile_n=96, tile_k=128,
                                       stages=4, cols=128, splits=0), **fields})
        if ok:
            dep.dep_projection_plan_set(plan, t)
            assert dep.dep_projection_plan_query(plan, 100).as_dict() == t.as_dict()
        else:
            with pytest.raises(dep.DepError):
                dep.dep_projection_plan_set(plan, t)
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_plan_save_format(dep, tmp_path):
    plan = dep.dep_projection_plan_host(49376, 7168, [1, 4, 8, 16], 152)
    try:
        path = str(tmp_path / "plan.txt")
        dep.dep_projection_plan_save(plan, path)
        lines = open(path).read().split("\n")
        assert lines[0] == "dep_projection_plan 2"
        assert lines[2] == "sms 152" and lines[3] == "shape 49376 7168" and lines[4] == "entries 4"
        rows = [list(map(int, l.split())) for l in lines[5:9]]
        table = dep.dep_projection_plan_table(plan)
        assert rows == [[t.max_rows, t.kind, t.ctas, t.tile_n, t.tile_k, t.stages, t.cols, t.splits]
                        for t in table]
    finally:
        dep.dep_projection_plan_destroy(plan)


def test_plan_load_rejects_bad_files(dep, tmp_path):
    p = tmp_path / "bad.txt"
    p.write_text("not a plan\n")
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_plan_load(str(p), 64, 64)
    assert e.value.status == dep.DEP_ERR_IO
    with pytest.raises(dep.DepError) as e:
        dep.dep_projection_plan_load(str(tmp_path / "missing.txt"), 64, 64)
    assert e.value.status == dep.DEP_ERR_IO


def test_status_strings(dep):
    for s in range(0, 9):
        assert dep.dep_status_string(s)
    assert dep.dep_status_string(1234) == "unknown status"


def test_k_piece_tactic_validation_and_save(dep, tmp_path):
    """The K-piece tensor-core kind: 1..64 pieces, 128-row tiles, 1/2/4 slices
    of 64 columns per stage; the piece count is rejected on every other kind and
    is written as the eighth field of a plan file entry."""
    plan = dep.dep_projection_plan_host(7168, 12288, [1, 16], 152)
    try:
        t = dep.dep_tactic_t(max_rows=16, kind=dep.DEP_KIND_TC_SPLIT, ctas=152, tile_n=128, tile_k=256,
                             stages=3, cols=16, splits=8)
        dep.dep_projection_plan_set(plan, t)
        q = dep.dep_projection_plan_query(plan, 9)
        assert (q.kind, q.splits, q.tile_k) == (dep.DEP_KIND_TC_SPLIT, 8, 256)
        for field, value in (("splits", 0), ("splits", 65), ("tile_n", 32), ("tile_k", 192),
                             ("stages", 1), ("cols", 24), ("stages", 12)):
            bad = dep.dep_tactic_t(**{**t.as_dict(), field: value})
            with pytest.raises(dep.DepError):
                dep.dep_projection_plan_set(plan, bad)
        fma = dep.dep_tactic_t(max_rows=3, kind=dep.DEP_KIND_SPLITK_FMA, ctas=152, tile_n=64, tile_k=256,
                               stages=4, cols=4, splits=2)
        with pytest.raises(dep.DepError):
            dep.dep_projection_plan_set(plan, fma)
        path = str(tmp_path / "plan.txt")
        dep.dep_projection_plan_save(plan, path)
        entries = [list(map(int, l.split())) for l in open(path).read().split("\n")[5:] if l]
        assert [16, dep.DEP_KIND_TC_SPLIT, 152, 128, 256, 3, 16, 8] in entries
    finally:
        dep.dep_projection_plan_destroy(plan)
