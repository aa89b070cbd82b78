"""Host-side pieces of bench.py that the JSON line depends on (no GPU needed)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_keeps_code_and_literals():
    src = 'int a = 1; // trailing\n/* block\n comment */ int b = 2;\nconst char *s = "x // not a comment";\n\n'
    out = bench.strip_comments(src)
    assert "trailing" not in out and "block" not in out
    assert "int a = 1;" in out and "int b = 2;" in out
    assert '"x // not a comment"' in out


def test_source_hash_ignores_comments_but_not_code():
    base = "__global__ void k(int *p) { p[0] = 1; }\n"
    assert bench.strip_comments("// note\n" + base) == bench.strip_comments(base)
    assert bench.strip_comments(base.replace("1", "2")) != bench.strip_comments(base)


def test_every_timed_kernel_has_a_source_hash():
    for kernel in bench.KERNEL_SOURCES:
        h = bench.kernel_source_hash(kernel)
        assert len(h) == 16 and int(h, 16) >= 0


def test_attention_kernel_choice_follows_head_dim():
    from programming_flashattention_fwd_gb300.inputs import ALL_WORKLOADS
    w128 = ALL_WORKLOADS["gqa_causal_b2_h32kv8_s4096"]
    w256 = ALL_WORKLOADS["gqa_causal_b2_h32kv8_s4096_d256"]
    assert bench.attention_kernel(w128, 0) == "fa::fa_fwd_kernel"
    assert bench.attention_kernel(w256, 0) == "fa::fa_fwd1_kernel"
    assert bench.attention_kernel(w128, 2) == "fa::fa_fwd1_kernel"
    assert bench.attention_kernel(w128, 3) == "fa::fa_fwd1_kernel"


def test_committed_profiles_name_kernel_workload_and_source():
    # every committed ncu summary names a kernel, a workload and the hash of the sources it
    # measured; the benchmark reports its traffic only while that hash matches the sources
    import glob
    import re
    from programming_flashattention_fwd_gb300.inputs import ALL_WORKLOADS
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        txt = open(path).read()
        kernel = re.search(r"^kernel: (\S+)$", txt, re.M).group(1)
        workload = re.search(r"^workload: (\S+)$", txt, re.M).group(1)
        sha = re.search(r"^kernel_source_sha: ([0-9a-f]{16})$", txt, re.M).group(1)
        assert kernel in bench.KERNEL_SOURCES, path
        assert re.search(r"^traffic_bytes_per_launch: \d+", txt, re.M), path
        if kernel.startswith("fa::fa_fwd"):
            assert workload in ALL_WORKLOADS, path
        fresh = sha == bench.kernel_source_hash(kernel)
        assert (bench.ncu_traffic(workload, kernel) is not None) == fresh, path


def test_suite_leads_with_the_largest_workload():
    from programming_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS
    # every benchmark configuration, plus the head-dim-256 workloads, each once
    assert set(WORKLOADS) <= set(bench.SUITE) <= set(WORKLOADS) | set(EXTRA_WORKLOADS)
    assert len(set(bench.SUITE)) == len(bench.SUITE)
    assert any(WORKLOADS.get(n) is None and EXTRA_WORKLOADS[n].D == 256 for n in bench.SUITE)
    head = WORKLOADS[bench.SUITE[0]]
    assert head.flops() == max(w.flops() for w in WORKLOADS.values())
    # the metric's non-causal half is in the suite
    assert any(not WORKLOADS[n].causal and WORKLOADS[n].D == 128 for n in bench.SUITE)
