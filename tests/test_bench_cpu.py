"""The benchmark's roofline numerator: the algorithmic KV bytes one decode step
reads, checked against a count built from the oracle's window regions and cache
row sizes, and against the per-workload totals derived separately for the
workload table (147.6 MB for the qwen3-4b layer, ...).  CPU only."""
import pytest

from int2_kv_cache_append_gb300 import synth as S
from oracle import oscar_oracle as O


@pytest.fixture(scope="module")
def bench():
    import bench as b  # argument parsing happens only in its main()
    return b


def _bytes_from_layout(w, T, v_bf16):
    # one (sequence, KV head): rows of each region times the row sizes of the
    # cache layout (a cache of one sequence and one KV head, capacity T)
    cfg = O.Config(1, 1, 1, 1, w.head_dim, w.sink, w.recent, max(T, 1),
                   flags=O.FLAG_V_BF16 if v_bf16 else 0)
    lay = O.layout(cfg)
    D = w.head_dim
    bf16_row = 2 * D
    int2_row = D // 4 + 4 * (D // O.GROUP)
    assert lay["codes_bytes"] >= lay["ncap"] * (D // 4)       # the row sizes the layout stores
    n_sink, tq, n_int, n_ring = O.regions(T, w.sink, w.recent)
    k = (n_sink + n_ring) * bf16_row + n_int * int2_row
    v = T * bf16_row if v_bf16 else k
    return k + v


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
@pytest.mark.parametrize("v_bf16", [False, True])
def test_kv_bytes_per_unit_match_the_layout(bench, name, v_bf16):
    w = S.WORKLOADS[name]
    for T in (1, w.sink, w.sink + 1, w.sink + w.recent, w.sink + w.recent + 1, w.context // 2, w.context):
        if T < 1:
            continue
        assert bench.kv_bytes_per_bh(w, T, v_bf16) == _bytes_from_layout(w, T, v_bf16), T


@pytest.mark.parametrize("name,total,unit", [
    ("tiny", 0.21e6, 0.01e6), ("qwen3-4b-layer", 147.6e6, 0.1e6), ("qwen3-8b-36L", 23.04e9, 0.01e9),
    ("hd512", 748e6, 1e6), ("qwen3-32b-decode", 76.6e6, 0.1e6)])
def test_step_totals_match_the_workload_table(bench, name, total, unit):
    # the table prints each total to the unit given: agreement within half of it
    w = S.WORKLOADS[name]
    got = bench.kv_bytes_per_bh(w, w.context) * w.batch * w.num_kv_heads * w.num_layers
    assert abs(got - total) <= unit / 2, got
