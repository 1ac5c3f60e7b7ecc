"""Host-side FLOP accounting of bench.py's block-masked runs, checked by brute
force on small shapes."""
import numpy as np
import pytest

import bench


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S", [1, 128, 300])
def test_visible_keys_brute_force(S, causal):
    nt = (S + 127) // 128
    m = np.random.default_rng(S).integers(0, 2, (2, nt, nt)).astype(np.uint8)
    vk = bench.visible_keys(m, S, causal)
    for h in range(2):
        for i in range(S):
            want = sum(1 for j in range(S) if m[h, i // 128, j // 128] and (not causal or j <= i))
            assert vk[h, i] == want


def test_all_ones_mask_counts_every_visible_pair():
    S = 1000
    m = np.ones((1, 8, 8), np.uint8)
    assert np.array_equal(bench.visible_keys(m, S, True)[0], np.arange(1, S + 1))
    assert np.all(bench.visible_keys(m, S, False)[0] == S)


def test_host_cpu_names_x86_and_arm_hosts(tmp_path):
    import bench
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Some Xeon @ 2.70GHz\n")
    assert bench.host_cpu(str(x86)).endswith("Some Xeon @ 2.70GHz")
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\n"
                   "CPU variant\t: 0x0\nCPU part\t: 0xd4f\nCPU revision\t: 0\n")
    assert bench.host_cpu(str(arm)).endswith("implementer 0x41 part 0xd4f")
    assert bench.host_cpu(str(tmp_path / "missing")) != ""


def test_sources_hash_ignores_comments_and_layout_only():
    """The DRAM-traffic records are keyed by a hash of the kernel code without
    comments: a comment or whitespace edit keeps the key, a code edit changes it."""
    base = "int f(int x) {\n    // doubles x\n    return 2 * x; /* no overflow check */\n}\n"
    comment_edit = "int f(int x) {\n    // doubles its argument\n    return 2 * x;\n}\n"
    layout_edit = "int f(int x) { return 2 * x; }\n"
    code_edit = "int f(int x) {\n    // doubles x\n    return 3 * x;\n}\n"
    assert bench._code_only(base) == bench._code_only(comment_edit) == bench._code_only(layout_edit)
    assert bench._code_only(base) != bench._code_only(code_edit)


def test_traffic_records_are_well_formed():
    """Every record line holds a 16-digit sources key, a workload name and a
    positive byte count."""
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "dram_traffic.txt")
    rows = [line.split() for line in open(path) if line.strip() and not line.startswith("#")]
    assert rows and all(len(r) == 3 and len(r[0]) == 16 and int(r[2]) > 0 for r in rows)
