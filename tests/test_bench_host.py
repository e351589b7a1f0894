"""Host-side logic of the benchmark, without a GPU: the byte accounting behind
the weight-bandwidth metric ("Strata" PR #2207 mmvq_bench table: weight
bytes of the matrix over the call time; PR #2746: grouped calls count the
experts actually read), the workload definitions, and the rule that a
committed ncu summary taken on other kernel sources is not used."""
import pytest

import bench
from block_quantized_matvec_gb300 import metrics


def test_block_sizes_follow_the_formats():
    # Q6_K: ql[128] + qh[64] + scales[16] + fp16 d; Q4_K: fp16 d, dmin + 12
    # packed scale/min bytes + qs[128]; Q5_K adds qh[32] to Q4_K
    assert metrics.BYTES_PER_256["q6_k"] == 128 + 64 + 16 + 2
    assert metrics.BYTES_PER_256["q4_k"] == 2 + 2 + 12 + 128
    assert metrics.BYTES_PER_256["q5_k"] == 2 + 2 + 12 + 32 + 128
    for planar in ("q6_k_planar", "q4_k_planar", "q5_k_planar"):
        assert metrics.BYTES_PER_256[planar] == metrics.BYTES_PER_256[planar[:4]]


def test_weight_bytes_of_the_pages_matrices():
    assert metrics.weight_bytes("q6_k", 10240, 2560) == 21_504_000      # "21.5 MB"
    assert metrics.weight_bytes("q6_k", 2560, 2560) == 5_376_000        # "5.38 MB"
    assert metrics.weight_bytes("q6_k_planar", 151936, 2560) == 319_065_600
    assert metrics.weight_bytes("q4_k", 12288, 2560) == 17_694_720
    with pytest.raises(ValueError):
        metrics.weight_bytes("q6_k", 16, 300)


def test_call_bytes_add_the_columns_and_outputs_once():
    w = metrics.weight_bytes("q6_k", 2560, 10240)
    for ncols in (1, 8):
        assert metrics.call_bytes("q6_k", 2560, 10240, ncols) == \
            w + ncols * (10240 // 32) * 36 + ncols * 2560 * 4


def test_moe_step_bytes_count_each_distinct_expert_once():
    per_expert = 2_211_840 + 1_105_920          # gate|up 1536 x 2560 and down 2560 x 768, Q4_K
    assert metrics.moe_step_bytes(1, 2560, 768) == per_expert
    assert metrics.moe_step_bytes(57, 2560, 768) == 57 * per_expert


@pytest.mark.parametrize("name", ["q6k_sweep", "q6k_sweep_gguf", "lm_head", "q4k_dense",
                                  "q5k_dense", "q4k_dense_gguf"])
def test_dense_workloads_are_valid_calls(name):
    cases = bench.workload_cases(name)
    assert cases
    for fmt, rows, K, cols in cases:
        assert fmt in metrics.BYTES_PER_256 and rows >= 1 and K % 256 == 0
        assert cols and all(1 <= c <= 8 for c in cols)


def test_the_default_workload_is_the_pages_sweep():
    cases = bench.workload_cases("q6k_sweep")
    assert sorted((r, k) for _, r, k, _ in cases) == [(2560, 2560), (2560, 10240), (10240, 2560)]
    assert all(cols == [1, 2, 4, 6, 8] for _, _, _, cols in cases)


def test_a_summary_from_other_kernel_sources_is_not_used(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "HERE", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc123")
    f = tmp_path / "profiles" / "x.md"
    f.write_text("# summary\n\ntraffic_bytes_per_mmvq_launch: 10871204\nkernel_source_sha256: abc123\n")
    assert bench.profiled_traffic("x.md") == 10871204
    f.write_text("# summary\n\ntraffic_bytes_per_mmvq_launch: 10871204\nkernel_source_sha256: ffff\n")
    assert bench.profiled_traffic("x.md") is None
    assert bench.profiled_traffic("missing.md") is None
