"""GPU score + Top-K against the oracle on hand-shaped inputs that exercise
the select's two paths (candidates gathered on chip, or refinement passes
when the threshold bin is too crowded), ties, ragged tiles and row groups."""
import numpy as np
import pytest

from oracle.indexer import score_topk
from synth.rng import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(keys_list, q, w, K, streams=None):
    """keys_list: per unit bf16 bits [L_u, 64]; q: bf16 bits [U, R, 8, 64]; w: [U, R, 8].
    With `streams` = (score stream, select stream), dsa_score and
    dsa_topk_select run there, ordered by dsa_stream_wait_stream."""
    import torch
    from decode_attention_dsa_gb300 import abi
    from decode_attention_dsa_gb300.units import UnitSet
    U = len(keys_list)
    R = q.shape[1]
    lmax = max(k.shape[0] for k in keys_list) + 8
    g = UnitSet(U, 4, lmax, mirror="device")
    for u, k in enumerate(keys_list):
        g.set_keys(u, 0, k)
    g.init([k.shape[0] for k in keys_list], abi.WARM_EMPTY)
    ws_b = abi.dsa_score_topk_workspace(U, R, lmax)
    ws = torch.zeros(ws_b, dtype=torch.uint8, device="cuda")
    out = torch.empty((U, R, K), dtype=torch.int32, device="cuda")
    qt = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda()
    wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    for _ in range(2):          # twice: the workspace must come back clean
        out.fill_(-5)
        if streams is None:
            abi.dsa_score_topk(g.units, U, R, K, qt, wt, out, lmax, ws, ws_b, g.dev_err)
        else:
            cur = torch.cuda.current_stream()
            abi.dsa_stream_wait_stream(streams[0], cur)
            abi.dsa_score(g.units, U, R, K, qt, wt, lmax, ws, ws_b, g.dev_err, streams[0])
            abi.dsa_stream_wait_stream(streams[1], streams[0])
            abi.dsa_topk_select(g.units, U, R, K, out, lmax, ws, ws_b, g.dev_err, streams[1])
            abi.dsa_stream_wait_stream(cur, streams[1])
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for u, k in enumerate(keys_list):
            _, want = score_topk(k, q[u], w[u], K)
            assert np.array_equal(got[u], want), f"unit {u}"
    assert g.check() == 0
    g.close()


def _bits(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_all_scores_equal_takes_lowest_positions():
    rng = np.random.default_rng(0)
    keys = [_bits(rng.integers(-4, 5, size=(40000, 64)))]
    q = _bits(np.zeros((1, 1, 8, 64)))
    _run(keys, q, np.ones((1, 1, 8)), 2048)


def test_few_distinct_values_many_ties():
    rng = np.random.default_rng(1)
    keys = [_bits(rng.integers(0, 2, size=(30000, 64))) for _ in range(2)]
    q = _bits(np.ones((2, 2, 8, 64)))
    q[:, :, :, 5:] = _bits(np.zeros(1))[0]
    _run(keys, q, np.ones((2, 2, 8)), 1000)


def test_long_ragged_history_three_rows():
    rng = np.random.default_rng(2)
    keys = [_bits(rng.integers(-4, 5, size=(131072 + 77, 64)))]
    q = _bits(rng.integers(-4, 5, size=(1, 3, 8, 64)))
    w = rng.integers(1, 5, size=(1, 3, 8))
    _run(keys, q, w, 2048)


def test_six_rows_two_row_groups_and_unequal_units():
    rng = np.random.default_rng(3)
    keys = [_bits(rng.integers(-4, 5, size=(n, 64))) for n in (5000, 12345, 300)]
    q = _bits(rng.integers(-4, 5, size=(3, 6, 8, 64)))
    w = rng.integers(1, 5, size=(3, 6, 8))
    _run(keys, q, w, 512)


def test_negative_weights_and_fractional_queries():
    rng = np.random.default_rng(4)
    keys = [_bits(rng.integers(-4, 5, size=(20000, 64)))]
    q = _bits(rng.integers(-64, 65, size=(1, 2, 8, 64)) / 16.0)
    w = rng.integers(-4, 5, size=(1, 2, 8))
    _run(keys, q, w, 777)


def test_many_selected_keys_in_one_cluster_range():
    """Most of a large Top-K lies in the first CTA's part of the history, so
    that CTA's ordered list of keys at or above the threshold bin overflows
    and the output is compacted from its whole range instead."""
    rng = np.random.default_rng(5)
    k = np.zeros((40000, 64))
    k[:6000] = rng.integers(1, 5, size=(6000, 64))
    keys = [_bits(k)]
    q = _bits(np.ones((1, 1, 8, 64)))
    _run(keys, q, np.ones((1, 1, 8)), 4096)


def test_short_history_in_few_tiles_and_empty_cluster_ranges():
    rng = np.random.default_rng(6)
    keys = [_bits(rng.integers(-4, 5, size=(n, 64))) for n in (2049, 2051, 4100, 9)]
    q = _bits(rng.integers(-4, 5, size=(4, 1, 8, 64)))
    w = rng.integers(1, 5, size=(4, 1, 8))
    _run(keys, q, w, 2048)


@pytest.mark.parametrize("R", [1, 2])
def test_more_units_than_score_ctas(R):
    """More units than the persistent score grid holds CTAs (4 per SM on the
    whole device): the grid cuts the flattened (unit, tile) space evenly, so
    CTAs cross unit boundaries (the query operand alternates between its two
    buffers, the shared histogram is flushed at each unit change). Ragged
    histories of 1 to 4 tiles, some shorter than K (every position kept)."""
    rng = np.random.default_rng(21 + R)
    lens = rng.integers(40, 520, size=700)
    keys = [_bits(rng.integers(-4, 5, size=(int(n), 64))) for n in lens]
    q = _bits(rng.integers(-4, 5, size=(700, R, 8, 64)))
    w = rng.integers(1, 5, size=(700, R, 8))
    _run(keys, q, w, 64)


@pytest.mark.parametrize("R", [1, 3])
def test_more_units_than_score_ctas_on_a_partition(R):
    """The same on an SM partition (five CTAs per SM): 200 units on the first
    partition of a split at 8 SMs (its 32 SMs hold 160 CTAs)."""
    from decode_attention_dsa_gb300 import abi
    rng = np.random.default_rng(31 + R)
    lens = rng.integers(200, 3000, size=200)
    keys = [_bits(rng.integers(-4, 5, size=(int(n), 64))) for n in lens]
    q = _bits(rng.integers(-4, 5, size=(200, R, 8, 64)))
    w = rng.integers(1, 5, size=(200, R, 8))
    first, second = abi.dsa_partition_split(8)
    try:
        _run(keys, q, w, 256, streams=(abi.dsa_partition_stream(first), abi.dsa_partition_stream(second)))
    finally:
        abi.dsa_partition_destroy(first)
        abi.dsa_partition_destroy(second)


@pytest.mark.parametrize("min_sms", [8, 96])
def test_score_and_select_on_two_sm_partitions(min_sms):
    """dsa_score on the first of two SM partitions (its persistent grid sized
    to the partition's SMs, whole CTAs per unit where the grid holds one per
    unit) and dsa_topk_select (8-CTA clusters) on the second: the same Top-K
    as the oracle, for units of unequal, ragged lengths."""
    import torch
    from decode_attention_dsa_gb300 import abi
    rng = np.random.default_rng(11)
    keys = [_bits(rng.integers(-4, 5, size=(n, 64))) for n in (70001, 257, 33333, 128, 90000)]
    q = _bits(rng.integers(-4, 5, size=(5, 2, 8, 64)))
    w = rng.integers(1, 5, size=(5, 2, 8))
    first, second = abi.dsa_partition_split(min_sms)
    try:
        n1, n2 = abi.dsa_partition_sms(first), abi.dsa_partition_sms(second)
        assert n1 >= min_sms and n2 >= 8
        assert n1 + n2 == torch.cuda.get_device_properties(0).multi_processor_count
        _run(keys, q, w, 2048, streams=(abi.dsa_partition_stream(first), abi.dsa_partition_stream(second)))
    finally:
        abi.dsa_partition_destroy(first)
        abi.dsa_partition_destroy(second)
