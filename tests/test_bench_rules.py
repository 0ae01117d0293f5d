"""The bench's roofline byte counts against the per-step figures of the hot-path
measurement table: U_k + W_2 per draft step is 97.2 MB (qwen4b), 155.6 MB (heavy),
198.6 MB (prod, V = 129280) and 116.7 MB (rnn).  The bench adds the gathered W_1
rows, h_k and w, which must stay a small correction; the strict per-cycle count
reads W_2 once for all gamma steps."""
import pytest

import bench
from speculative_decoding_drafter_markov_gb300 import workloads as W

TABLE_MB = {"qwen4b": 97.2, "heavy": 155.6, "prod": 198.6, "rnn": 116.7}


@pytest.mark.parametrize("name", sorted(TABLE_MB))
def test_step_bytes_match_the_table(name):
    wl = W.WORKLOADS[name]
    step = bench.draft_step_bytes(wl)
    extras = (wl.R * wl.r + wl.R * wl.d) * 2 + (wl.d + wl.r) * 4  # W_1 rows, h_k (bf16), w (fp32)
    assert abs((step - extras) / 1e6 - TABLE_MB[name]) < 0.05
    assert extras / step < 0.03  # h_k dominates: 2.2 % at prod (d = 4096, R = 512)


@pytest.mark.parametrize("name", sorted(TABLE_MB))
def test_strict_cycle_reads_w2_once(name):
    wl = W.WORKLOADS[name]
    w2 = wl.V * wl.r * 2
    per_step = bench.draft_step_bytes(wl)
    assert bench.draft_cycle_bytes_strict(wl) == wl.gamma * (per_step - w2) + w2


def test_qwen4b_figures_quoted_by_the_bench():
    wl = W.WORKLOADS["qwen4b"]
    assert wl.gamma * bench.draft_step_bytes(wl) == 780886016  # per launch, W_2 counted each step
    assert bench.draft_cycle_bytes_strict(wl) == 236347392


def test_training_loss_bytes():
    B, gamma, V = bench.TRAIN["B"], bench.TRAIN["gamma"], bench.TRAIN["V"]
    N = B * gamma
    logits_once = 2 * N * V * 2  # draft and target rows, bf16
    gradient_once = N * V * 4    # fp32
    assert logits_once + gradient_once <= bench._train_bytes() < (logits_once + gradient_once) * 1.0001
    assert abs(bench._train_bytes() / 1e6 - 622.3) < 0.1


def test_verify_bytes_follow_the_table():
    # every drafted token verified at qwen4b: 576 target rows (175 MB), then per
    # request a target row and, when it rejected, its U row, plus W_2 -- at most
    # the table's 116.7 MB of residual rows
    wl = W.WORKLOADS["qwen4b"]
    rows = wl.R * (wl.gamma + 1)
    lo = bench.verify_cycle_bytes(wl, rows, 0)
    hi = bench.verify_cycle_bytes(wl, rows, wl.R)
    assert abs(rows * wl.V * 2 / 1e6 - 175.0) < 0.1
    assert abs((hi - rows * wl.V * 2) / 1e6 - 116.7) < 0.1
    assert hi - lo == wl.R * wl.V * 2


def test_verify_roofline_arithmetic():
    wl = W.WORKLOADS["qwen4b"]
    steps, rejected, verified = 4, 4 * 60, 4 * wl.R * wl.gamma
    r = bench._verify_roofline(wl, verified, rejected, steps, [0.0829] * steps, 6761.6)
    nbytes = bench.verify_cycle_bytes(wl, wl.R * (wl.gamma + 1), 60)
    assert r["algorithmic_bytes_per_cycle"] == nbytes
    assert abs(r["achieved"] - nbytes / 82.9e-6 / 1e9) < 1e-6 * r["achieved"]
    assert abs(r["frac"] - r["achieved"] / 6761.6) < 1e-12


def test_verify_roofline_without_timings():
    wl = W.WORKLOADS["qwen4b"]
    assert bench._verify_roofline(wl, 8, 1, 1, [], 6761.6) is None
    assert bench._verify_roofline(wl, 8, 1, 1, [0.0], 6761.6) is None


def test_verify_strict_bytes_drop_the_second_read():
    wl = W.WORKLOADS["prod"]
    rows = wl.R * 5
    assert (bench.verify_cycle_bytes(wl, rows, 100) - bench.verify_cycle_bytes(wl, rows, 100, reread=False)
            == wl.R * wl.V * 2)
    r = bench._verify_roofline(wl, 4 * wl.R * 4, 400, 4, [0.2] * 4, 6761.6)
    assert r["frac_strict"] < r["frac"]


def test_traffic_record_keyed_by_source_hash(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("draft_step_tc")
    rec = tmp_path / "rec.txt"
    rec.write_text(f"# comment\ndraft_step_tc prod {h} 100 20 full-size\n"
                   "draft_step_tc heavy 0000000000000000 5 5 full-size\n")
    monkeypatch.setattr(bench, "NCU_DRAM_FILE", str(rec))
    assert bench.ncu_traffic("draft_step_tc", "prod")[0] == 120
    assert bench.ncu_traffic("draft_step_tc", "heavy")[0] is None  # stale: another kernel build
    assert bench.ncu_traffic("draft_step_tc", "qwen4b")[0] is None  # never captured
