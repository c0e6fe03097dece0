"""Top-K selection on its own: qsa_topk_select on synthetic score rows against
the oracle's exact top-K (score descending, block index ascending), bit-exact.

The score distributions cover every way the kernel can settle the K-th largest
key: spread scores (a short candidate list ranked directly), a narrow cluster
inside a wide range (a long candidate list refined by further passes, or, past
the candidate capacity, passes over the whole row), heavy ties and signed
zeros (ties taken by the lower block index, -0 equal to +0), and rows longer
than the kernel keeps in shared memory (keys read from global memory). Rows of
up to 16k blocks keep their keys in registers, longer rows up to about 45k
blocks in shared memory, and longer ones read them from global memory: the
cases below cover all three."""
import numpy as np
import pytest
import torch

from indexer_selected_sparse_gb300 import synth as S
from oracle import qsa_oracle as O

pytestmark = pytest.mark.gpu

Q = pytest.importorskip("indexer_selected_sparse_gb300.qsa")


def run_select(ratio, budget, ns, kind, seed):
    cfg = Q.Config(ratio, budget, 64, 128, 32, 4)
    K = cfg.topk
    ld = (max(ns) + 3) // 4 * 4
    scores = S.select_scores(seed, len(ns), ld, kind)
    # visible = n * ratio + (ratio - 1): the incomplete tail does not change n
    pos0 = torch.tensor([n * ratio + ratio - 2 for n in ns], dtype=torch.int32)
    rows = Q.Rows(torch.arange(len(ns), dtype=torch.int32, device="cuda"), pos0.cuda(), 1)
    sel = torch.full((len(ns), K), -7, dtype=torch.int32, device="cuda")
    nsel = torch.full((len(ns),), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.qsa_topk_select(cfg, rows, scores.cuda(), ld, sel, nsel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    sel = sel.cpu().numpy()
    nsel = nsel.cpu().numpy()
    for r, n in enumerate(ns):
        want = O.select_blocks(scores[r, :n].numpy().astype(np.float64), K)
        assert nsel[r] == len(want), (kind, n)
        assert np.array_equal(sel[r, : len(want)], want), (kind, n, r)
        assert (sel[r, len(want):] == -1).all()


@pytest.mark.parametrize("kind", S.SCORE_KINDS)
def test_select_k512_on_chip(kind):
    # K = 512; rows from just above K to 16384 blocks (64k tokens)
    run_select(4, 2048, [513, 600, 4000, 8192, 8193, 16384], kind, seed=21)


@pytest.mark.parametrize("kind", ["spread", "cluster", "few_values"])
def test_select_rows_beyond_shared_memory(kind):
    # ratio 2: 100000 blocks is more than the kernel stages on chip
    run_select(2, 1024, [100000, 45056, 45057], kind, seed=22)


@pytest.mark.parametrize("kind", ["spread", "relu_sum", "few_values"])
def test_select_very_long_rows_and_a_short_one_in_one_launch(kind):
    # 120000 and 60000 blocks read from global memory, 513 kept in registers
    run_select(2, 1024, [120000, 60000, 513], kind, seed=25)


@pytest.mark.parametrize("kind", ["spread", "nonneg", "cluster"])
def test_select_k2048(kind):
    run_select(4, 8192, [2049, 5000, 20000], kind, seed=23)


def test_select_dense_rows_take_every_block():
    # n <= K: every block, in order, padded with -1
    run_select(4, 2048, [1, 2, 511, 512], "spread", seed=24)


@pytest.mark.parametrize("kind", S.SCORE_KINDS)
def test_select_short_rows_split_over_the_cluster(kind):
    # rows of up to 16k blocks are split over four CTAs in runs of a multiple of
    # 4 blocks: at 17 or 18 blocks the last CTA holds none and the third one or
    # two; K = 16
    run_select(4, 64, [17, 18, 23, 31, 64, 100, 1000, 16383], kind, seed=26)


@pytest.mark.parametrize("kind", ["spread", "few_values", "signed_zero"])
def test_select_k1(kind):
    # K = 1: the single largest block, ties to the lowest index
    run_select(4, 4, [2, 3, 5, 4097, 9000, 20000, 32768], kind, seed=27)


@pytest.mark.parametrize("kind", ["spread", "cluster", "few_values", "relu_sum"])
def test_select_k2048_in_registers(kind):
    # K = 2048 with rows held in registers across the cluster
    run_select(4, 8192, [2049, 4100, 8192, 12000, 16384], kind, seed=28)


@pytest.mark.parametrize("kind", S.SCORE_KINDS)
def test_select_rows_past_a_layout_boundary(kind):
    # past 8192 blocks a thread holds its run of 8 keys plus one key from the
    # row's tail (ties there come after every tie of the runs), past 9216 runs
    # of 12, past 12288 runs of 16: each side of each boundary, K = 512
    run_select(4, 2048, [8193, 8200, 8256, 9215, 9216, 9217, 12288, 12289], kind, seed=29)


@pytest.mark.parametrize("kind", ["spread", "few_values", "signed_zero"])
def test_select_k2048_with_tail_keys(kind):
    run_select(4, 8192, [8193, 9000, 9216], kind, seed=30)


@pytest.mark.parametrize("kind", S.SCORE_KINDS)
def test_select_runs_of_32(kind):
    # past 16384 blocks (up to 32768) a thread's run is 32 keys, 16 in registers
    # and 16 in shared memory; 32769 takes the shared-memory path
    run_select(4, 2048, [16385, 20000, 24577, 32767, 32768, 32769], kind, seed=31)


@pytest.mark.parametrize("kind", ["spread", "few_values", "cluster"])
def test_select_runs_of_32_k2048(kind):
    run_select(4, 8192, [16385, 30000, 32768], kind, seed=32)


def test_select_all_equal_rows_take_the_lowest_indices():
    # a row whose scores are all equal has an empty key range: every layout
    # (runs of 4 .. 32, the shared-memory path) takes the K lowest block indices
    cfg = Q.Config(4, 2048, 64, 128, 32, 4)
    K = cfg.topk
    ns = [600, 8193, 12000, 16384, 20000, 32768, 40000]
    ld = (max(ns) + 3) // 4 * 4
    scores = torch.full((len(ns), ld), 2.5, dtype=torch.float32)
    scores[1, :] = -0.0  # signed zeros compare equal to +0
    scores[1, ::3] = 0.0
    pos0 = torch.tensor([n * 4 + 2 for n in ns], dtype=torch.int32)
    rows = Q.Rows(torch.arange(len(ns), dtype=torch.int32, device="cuda"), pos0.cuda(), 1)
    sel = torch.full((len(ns), K), -7, dtype=torch.int32, device="cuda")
    nsel = torch.full((len(ns),), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.qsa_topk_select(cfg, rows, scores.cuda(), ld, sel, nsel, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    sel = sel.cpu().numpy()
    for r, n in enumerate(ns):
        want = O.select_blocks(scores[r, :n].numpy().astype(np.float64), K)
        assert np.array_equal(want, np.arange(K))
        assert nsel[r].item() == K and np.array_equal(sel[r], want), (r, n)


@pytest.mark.parametrize("n_rows", [8, 40, 80])
@pytest.mark.parametrize("kind", ["spread", "few_values", "relu_sum", "infinite"])
def test_select_cluster_sizes_and_one_cta_layouts(n_rows, kind):
    # rows past 9216 blocks go to a cluster of 4 CTAs per row when 4 x rows
    # CTAs fit on the GPU (8 rows), of 2 when 2 x rows fit (40 rows), else (80
    # rows) to one CTA per row: runs of 12 or 16 register keys, runs of 32
    cycle = [9217, 12288, 12289, 16384, 16385, 20000, 32768, 513, 8193, 600, 30001]
    ns = [cycle[i % len(cycle)] for i in range(n_rows)]
    run_select(4, 2048, ns, kind, seed=33 + n_rows)
