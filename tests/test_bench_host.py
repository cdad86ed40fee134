"""Host-side pieces of bench.py that need no GPU: the comment-insensitive
source hash that gates the recorded ncu traffic, and the traffic table."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_layout():
    a = "int a = 1; // note\n/* block\n  comment */ int  b =\n 2;\n"
    b = "int a = 1;\nint b = 2;"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_keeps_literals_and_code_changes():
    src = 'asm("mov.u32 %0, 1; // not a comment" : "=r"(x)); char c = \'"\'; int y = 2;'
    out = bench._code_only(src)
    assert "// not a comment" in out and "int y = 2;" in out
    assert bench._code_only("int y = 2;") != bench._code_only("int y = 3;")


def test_traffic_row_gated_by_code_hash(tmp_path, monkeypatch):
    # a recorded row counts while the kernel's code is unchanged: a comment
    # edit keeps it, a code edit turns the field null
    import shutil
    src = os.path.join(ROOT, "exact_attention_attn_gb300", "csrc")
    dst = tmp_path / "exact_attention_attn_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["attn_tc2_kernel"]:
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    h = bench.kernel_source_hash("attn_tc2_kernel")
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        "| workload | kernel | source hash | bytes per launch |\n|---|---|---|---|\n"
        f"| wl | attn_tc2_kernel<128, true> | {h} | 12345 |\n")
    assert bench.recorded_traffic("wl") == (12345.0, "attn_tc2_kernel<128, true>")
    assert bench.recorded_traffic("other") == (None, None)
    k = dst / "attn_tc2.cu"
    k.write_text(k.read_text() + "\n// a comment added later\n")
    assert bench.recorded_traffic("wl")[0] == 12345.0
    k.write_text(k.read_text() + "\nstatic int later_code = 1;\n")
    assert bench.recorded_traffic("wl") == (None, None)


def test_oracle_leg_of_every_path():
    # each path's CPU leg runs one head of a tiny workload through its oracle
    # and credits that head's FLOPs (2.5 x the forward's for the backward)
    from exact_attention_attn_gb300.workloads import Workload, make_workload_inputs
    w = Workload("tiny_gqa_causal", B=1, Hq=2, Hkv=1, Nq=72, Nkv=72, D=64, causal=True, seed=5)
    q, k, v = make_workload_inputs(w)
    for path in bench.PATHS:
        extra = bench.path_host_inputs(path, w)
        tf, heads, dt, nrows = bench.time_oracle(w, q, k, v, budget_s=0.0, path=path, extra=extra)
        assert heads == 1 and nrows == w.Nq and tf > 0
        assert abs(tf * dt * 1e12 - (2.5 if path == "bwd" else 1.0) * w.flops() / 2) < 1e-6 * w.flops()
        assert f"1 (b,hq) heads" in bench.oracle_sample_text(w, heads, dt, nrows, 1, path) or path == "fwd"


def test_mask_store_is_padded_to_eight_columns():
    # the masked path's mask is a [Nq, Nkv] view of a store whose rows are
    # multiples of 8 elements (16 bytes), as attn_fwd_masked requires
    from exact_attention_attn_gb300.workloads import Workload
    w = Workload("tiny", B=1, Hq=1, Hkv=1, Nq=5, Nkv=13, D=64, causal=False, seed=1)
    m = bench.path_host_inputs("mask", w)["mask"]
    assert tuple(m.shape) == (5, 13) and m.stride() == (16, 1)
    assert set(bench.path_host_inputs("bwd", w)) == {"dout"} and bench.path_host_inputs("fwd", w) == {}
