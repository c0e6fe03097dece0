"""The seeded input generator: the hash against its published definition,
position-addressability (any row regenerates on its own), and the value
distributions the workloads call for."""
import numpy as np
import torch

from indexer_selected_sparse_gb300 import synth as S


def lowbias32_python(x):
    # Chris Wellons' lowbias32, written with Python integers
    x ^= x >> 16
    x = (x * 0x7FEB352D) & 0xFFFFFFFF
    x ^= x >> 15
    x = (x * 0x846CA68B) & 0xFFFFFFFF
    x ^= x >> 16
    return x


def test_hash_matches_definition():
    xs = [0, 1, 2, 0xFFFFFFFF, 0x80000000, 123456789, 0xDEADBEEF] + list(range(1000, 1100))
    got = S.hash32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert got == [lowbias32_python(x) for x in xs]


def test_rows_regenerate_independently():
    sh = S.SHAPES_MAIN
    k, v, i = S.token_rows(sh, 1, 5, torch.arange(100, 140))
    k2, v2, i2 = S.token_rows(sh, 1, 5, torch.tensor([117, 103]))
    assert torch.equal(k[17], k2[0]) and torch.equal(v[3], v2[1]) and torch.equal(i[17], i2[0])
    # a different epoch (fresh rows after a rewind) gives different values
    k3, _, _ = S.token_rows(sh, 1, 5, torch.arange(100, 140), epoch=1)
    assert not torch.equal(k, k3)


def test_distributions():
    sh = S.SHAPES_MAIN
    k, v, i = S.token_rows(sh, 2, 0, torch.arange(0, 512))
    kf = k.float()
    assert abs(kf.mean().item()) < 0.01 and abs(kf.var().item() - 1.0) < 0.02
    assert kf.abs().max().item() <= 6.0
    assert set(i.float().unique().tolist()) == set(float(x) for x in range(-8, 9))
    q, qi, w = S.query_rows(sh, 2, 0, torch.arange(0, 64))
    assert set(w.unique().tolist()) == {0.25, 0.5, 1.0, 2.0}
    assert qi.float().abs().max().item() == 8.0


def test_page_table_is_a_permutation():
    pt = S.page_table(1, 4, 100, contiguous=False)
    assert sorted(pt.reshape(-1).tolist()) == list(range(400))
    assert not torch.equal(pt.reshape(-1), torch.arange(400, dtype=torch.int32))
    assert torch.equal(S.page_table(1, 4, 100, contiguous=True).reshape(-1),
                       torch.arange(400, dtype=torch.int32))


def test_ragged_prefixes_cover_the_boundary():
    p = S.workload(3).prefixes
    assert len(p) == 64 and {2050, 2051, 2052} <= set(p)
    assert min(p) >= 512 and max(p) <= 131072
    assert sum(1 for x in p if x < 2050) >= 3 and sum(1 for x in p if x > 8192) >= 20


def test_select_scores_kinds_are_seeded_and_shaped():
    for kind in S.SCORE_KINDS:
        a = S.select_scores(5, 3, 257, kind)
        b = S.select_scores(5, 3, 257, kind)
        assert a.shape == (3, 257) and a.dtype == torch.float32
        assert torch.equal(a, b) and not torch.isnan(a).any()
        assert torch.isfinite(a).all() or kind == "infinite"
    inf = S.select_scores(5, 2, 8192, "infinite")
    assert (inf == float("inf")).sum() > 600 and (inf == float("-inf")).sum() > 100
    z = S.select_scores(5, 2, 4096, "signed_zero")
    assert (torch.signbit(z) & (z == 0)).any() and (~torch.signbit(z) & (z == 0)).any()
    c = S.select_scores(5, 2, 4096, "cluster")
    assert c.max() > 1e29 and c.min() < -1e29
