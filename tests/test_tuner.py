"""bench.py's tuner, host side (no GPU): the rule that keeps a tabled choice
within run-to-run noise, the dispatch table's write / read round trip, and
that every launch choice the tuner times is a plan the planner accepts with
the path it asks for."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import w4a8_quantized_serving_qoq_gb300 as qoq  # noqa: E402

SMS = 152


def test_pick_choice_keeps_a_tabled_choice_within_the_noise_band():
    t = {"a": 100.0, "b": 100.4, "c": 101.0}
    assert bench.pick_choice(t, None) == "a"
    assert bench.pick_choice(t, "b") == "b"    # 0.4 % slower than the fastest: kept
    assert bench.pick_choice(t, "c") == "a"    # 1 % slower: replaced
    assert bench.pick_choice(t, "gone") == "a"  # no longer a candidate
    edge = {"a": 100.0, "b": 100.0 * (1.0 + bench.TUNE_KEEP_FRAC)}
    assert bench.pick_choice(edge, "b") == "b"
    past = {"a": 100.0, "b": 100.0 * (1.0 + 2 * bench.TUNE_KEEP_FRAC)}
    assert bench.pick_choice(past, "b") == "a"


def test_dispatch_table_write_read_round_trip(tmp_path, monkeypatch):
    entries = [
        dict(N=28672, K=4096, group=0, M=4096, path=1, bt=128, ctas=152, sched=2, us=580.0, rule_us=584.2),
        dict(N=4096, K=4096, group=128, M=1, path=3, bt=0, ctas=8, sched=0, us=4.25, rule_us=4.25),
        dict(N=6144, K=4096, group=128, M=8, path=2, bt=16, ctas=144, sched=0, us=9.57, rule_us=9.53),
    ]
    monkeypatch.setattr(bench, "DISPATCH_TABLE", str(tmp_path / "table.inc"))
    bench.write_dispatch_table(entries, SMS)
    assert bench.read_dispatch_table() == {
        (e["N"], e["K"], e["group"], e["M"]): (e["path"], e["bt"], e["ctas"], e["sched"]) for e in entries}
    rows = [l for l in open(tmp_path / "table.inc") if l.startswith("{")]
    assert [r.split(",")[:4] for r in rows] == [["{4096", " 4096", " 128", " 1"], ["{6144", " 4096", " 128", " 8"],
                                                ["{28672", " 4096", " 0", " 4096"]]
    assert all(r.split(",")[4].strip() == str(SMS) for r in rows)


def test_committed_table_holds_only_tuner_candidates():
    """Each measured entry is one of the choices the tuner times for its shape."""
    table = bench.read_dispatch_table()
    assert table
    for (N, K, group, M), choice in table.items():
        assert choice in bench.gemm_candidates(M, N, K, group, SMS), (N, K, group, M, choice)


SHAPES = [((6144, 4096), 128), ((4096, 4096), 128), ((28672, 4096), 128), ((4096, 14336), 128),
          ((59136, 8192), 128), ((8192, 29568), 128), ((28672, 4096), 0)]


@pytest.mark.parametrize("NK,group", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096])
def test_every_tuning_candidate_is_a_plan_of_its_path(NK, group, M):
    N, K = NK
    cands = bench.gemm_candidates(M, N, K, group, SMS)
    assert cands[0] == (0, 0, 0, 0) and len(set(cands)) == len(cands)
    for path, bt, ctas, sched in cands:
        opt = qoq.gemm_options(kernel=path, tokens_per_tile=bt, num_ctas=ctas, schedule=sched)
        p = qoq.qoq_gemm_plan(M, N, K, group, SMS, opt)
        if path:
            assert p["path"] == path, (path, bt, ctas, sched)
        if path in (1, 2):
            assert p["tokens_per_tile"] == bt and p["num_ctas"] == min(ctas, p["k_stages"])
        if path == 3:
            # the cluster size asked for, or the next larger one whose CTAs'
            # activation slices fit in shared memory (K = 29568 at 8 tokens)
            csize = p["num_ctas"] // (N // 128)
            assert p["num_ctas"] == (N // 128) * csize and csize in (1, 2, 4, 8) and csize >= ctas
            if csize > ctas:  # the requested size's slice is well above 128 KB
                assert M * K // ctas > 128 * 1024
