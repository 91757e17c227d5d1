"""Host-side pieces of bench.py (no GPU): the profile staleness hash and the
algorithmic byte counts the roofline divides by."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_inputs as mi  # noqa: E402


def test_code_hash_ignores_comments_and_layout():
    a = "int f(int x) {  // one\n  return x + 1; /* two\n three */ }\n"
    b = "int f(int x)\n{\n    return x + 1;\n}\n// a trailing note\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_profile_traffic_counts_only_for_the_current_kernel(tmp_path):
    # an ncu summary carries the hash of the kernel code it was taken on; a
    # profile of other code gives no traffic figure
    cur = bench.kernel_source_sha("experts")
    (tmp_path / "experts_w1.md").write_text(f"dram_bytes_per_launch: 1234\nsource_sha: {cur}\n")
    (tmp_path / "experts_w2.md").write_text("dram_bytes_per_launch: 1234\nsource_sha: 000000000000\n")
    assert bench.profiled_traffic("experts", "w1", str(tmp_path)) == 1234.0
    assert bench.profiled_traffic("experts", "w2", str(tmp_path)) is None
    assert bench.profiled_traffic("experts", "no_such_workload", str(tmp_path)) is None


def test_committed_profiles_carry_traffic_and_hash():
    for workload in ("verify_latent_s8", "verify_s32"):
        txt = open(os.path.join(ROOT, "profiles", f"experts_{workload}.md")).read()
        assert "dram_bytes_per_launch:" in txt and "source_sha:" in txt


def test_algorithmic_bytes_per_expert():
    # one touched expert: 3 I d e2m1 codes (half a byte each) and 3 I d / 32
    # e8m0 scales = 3 I d 17/32 bytes; 3,342,336 B at d = 4096, I = 512
    cfg = mi.CONFIGS[1]
    alg = bench.algorithmic_bytes(cfg, 1)
    assert alg["experts"] == 3 * cfg.I * cfg.d * 17 // 32 == 3342336
    assert alg["step"] == alg["experts"] + cfg.E * cfg.d * 2 + 4 * cfg.E


def test_ktrace_cli_parses():
    """The trace-timeline tool's command line (the tool itself needs a GPU)."""
    import pytest
    from mxfp4_mixture_experts_route_gb300 import ktrace
    with pytest.raises(SystemExit) as e:
        ktrace.main(["--help"])
    assert e.value.code == 0
