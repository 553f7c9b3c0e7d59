"""Host-side pieces of bench.py that need no GPU: the oracle baseline of the
ReTopK leg (its FIFO built from the oracle's own exact prefill supports, its
steps timed per path class) on a downsized stream."""
import re


def test_retopk_oracle_baseline_sample():
    import bench
    from workloads.gen import make_retopk
    wl = make_retopk(L0=3000, steps=24, K=32, C=4, R=2, W=4, T_r=8)
    r = bench.oracle_retopk_baseline(wl, budget_s=60.0)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["unit"] == bench.UNIT
    assert r["value"] > 0
    m = re.search(r"steps 0-(\d+) of the stream \((\d+) exact at .* (\d+) reuse at", r["sample"])
    assert m, r["sample"]
    last, n_exact, n_reuse = (int(x) for x in m.groups())
    # the whole downsized stream fits the budget; steps 0, 8 and 16 refresh
    assert last == wl.steps - 1 and n_exact + n_reuse == wl.steps
    assert n_exact >= 3 and n_reuse >= 1
