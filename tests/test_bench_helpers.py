"""The benchmark's host-side helpers that feed the roofline object: algorithmic bytes and FLOPs
of one attention launch, and the DRAM traffic read from a committed ncu summary, which must be
dropped (null) as soon as the profiled kernel's own sources change."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import mla_workloads as W  # noqa: E402


def test_decode_algorithmic_bytes_and_flops_match_the_hand_count():
    # B=16 sequences of 4096 tokens, 128 heads, rows of 576 bf16, latent 512
    case = {"shape": W.DEEPSEEK_V2, "seq_lens": np.full(16, 4096, dtype=np.int32)}
    b, f = bench.workload_numbers(case)
    per_seq = 4096 * 576 * 2 + 128 * 576 * 2 + 128 * (512 * 2 + 4)
    assert b == 16 * per_seq == 79962112
    assert f == 16 * 2 * 4096 * 128 * (576 + 512) == 18253611008


def test_prefill_flops_count_the_causal_triangle():
    T = 5
    case = {"shape": W.DEEPSEEK_V2, "seq_lens": np.array([T], dtype=np.int32), "T": T}
    b, f = bench.workload_numbers(case)
    pairs = sum(i + 1 for i in range(T))  # query i sees tokens 0..i
    assert f == 2 * 128 * (576 + 512) * pairs
    assert b == T * 576 * 2 + T * (128 * 576 * 2 + 128 * (512 * 2 + 4))


def test_source_digest_is_per_kernel():
    a = bench.source_digest("tc_attention")
    g = bench.source_digest("tc_gemm")
    assert a != g and a != bench.source_digest()
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "mla_latent_kv_79_b300", "csrc", f)), f


def test_code_text_drops_comments_only():
    src = "int a; // one\n/* two\n three */ int b;  \n\n  // four\nint c = 1 / 2;\n"
    assert bench.code_text(src) == "int a;\n int b;\nint c = 1 / 2;"
    # a comment edit keeps the digest, a code edit does not
    base = {f: "int x = 1; // note\n" for f in bench.KERNEL_SOURCES["tc_flash"]}
    d0 = bench.source_digest("tc_flash", read=lambda f: base[f])
    reworded = dict(base, **{"tc_flash.cuh": "int x = 1; // another note\n/* and more */\n"})
    changed = dict(base, **{"tc_flash.cuh": "int x = 2; // note\n"})
    assert bench.source_digest("tc_flash", read=lambda f: reworded[f]) == d0
    assert bench.source_digest("tc_flash", read=lambda f: changed[f]) != d0


def _write_profile(d, digest, nbytes=12345):
    p = d / "tc_attention_decode_b16_l4096.md"
    p.write_text(f"# capture\n\n- dram_bytes_per_launch: {nbytes}\n- source_digest: {digest} (of some files)\n")


def test_traffic_is_read_when_the_kernel_sources_match(tmp_path, monkeypatch):
    _write_profile(tmp_path, bench.source_digest("tc_attention"))
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench.ncu_traffic("tc_attention", "decode_b16_l4096") == 12345


def test_traffic_is_null_once_the_kernel_sources_changed(tmp_path, monkeypatch):
    _write_profile(tmp_path, "0123456789abcdef")
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench.ncu_traffic("tc_attention", "decode_b16_l4096") is None
    # and a missing summary is null too
    assert bench.ncu_traffic("tc_attention", "decode_long_b4") is None


@pytest.mark.parametrize("out_proj", [False, True])
def test_config_names_the_step(out_proj):
    case = {"shape": W.DEEPSEEK_V2, "seq_lens": np.full(16, 4096, dtype=np.int32)}
    c = bench.config_of("decode_b16_l4096", case, out_proj)
    assert c["workload"] == "decode_b16_l4096" and c["batch"] == 16 and c["seq_len"] == 4096
    assert ("W_O" in c["step"]) == out_proj


def test_oracle_heads_keep_all_heads_unless_the_float64_restore_would_not_fit():
    def heads(lens):
        return bench.oracle_heads({"shape": W.DEEPSEEK_V2, "seq_lens": np.array(lens)})
    assert heads([4096] * 16) == 128
    assert heads([256, 8192]) == 128
    h = heads([32768, 131072])
    assert h < 128 and 128 % h == 0 and h * 2 * 131072 * 128 * 8 <= 4 << 30


def test_oracle_sample_text_states_the_subset():
    case = {"shape": W.DEEPSEEK_V2, "seq_lens": np.array([300, 500, 700])}
    t = bench.oracle_sample_text(case, 2, 3, 16)
    assert "2 of 3 sequences" in t and "16 of 128 heads" in t and "scaled by 8" in t and "300-500" in t
    assert "all 128 heads" in bench.oracle_sample_text(case, 1, 3, 128)


@pytest.mark.parametrize("append", [False, True])
def test_cpu_oracle_sample_runs_on_a_head_subset(append):
    case = W.make_decode_case(W.TINY, "f32", [10, 70], seed=3, append=append)
    t_all = bench.cpu_oracle_sample(case, [0, 1], out_proj=True)
    t_two = bench.cpu_oracle_sample(case, [1], out_proj=False, heads=2)
    assert t_all > 0 and t_two > 0


def test_cpu_baseline_line_is_bounded_and_described():
    case = W.make_decode_case(W.TINY, "f32", [10, 70, 30], seed=4)
    line = bench.cpu_baseline(case, out_proj=False, budget_s=0.0)  # stops after one sequence
    assert line["kind"] == "oracle" and line["unit"] == bench.UNIT and line["value"] > 0
    assert line["cores"] >= 1 and "1 of 3 sequences" in line["sample"]
    full = bench.cpu_baseline(case, out_proj=True)
    assert "3 of 3 sequences" in full["sample"] and "all 4 heads" in full["sample"]
