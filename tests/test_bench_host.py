"""Host logic of bench.py (CPU): every workload names a kernel whose sources
exist, the algorithmic byte counts equal the sums worked out by hand from the
tensors each operation must read and write once, and a committed ncu summary
is only used for its traffic while the kernel's sources are unchanged."""
from __future__ import annotations

import os

import pytest

import bench
from fp8_activation_quantization_gb300 import synth


def test_every_workload_has_a_kernel_with_sources_and_an_input_set():
    csrc = os.path.join(bench.ROOT, "fp8_activation_quantization_gb300", "csrc")
    for name, kern in bench.KERNEL_OF.items():
        assert kern in bench.KERNEL_SOURCES, name
        for f in bench.KERNEL_SOURCES[kern]:
            assert os.path.exists(os.path.join(csrc, f)), (name, f)
        assert bench.SYNTH_OF.get(name, name) in synth.WORKLOADS, name
    assert bench.DEFAULT_WORKLOAD in bench.KERNEL_OF


# (workload, T, C, weighted, bytes): bf16 input 2 B, codes 1 B, scales 4 B per
# 128-group; the SwiGLU input is [T, 2H] with C = 2H columns.
CASES = [
    # plain: read 2TC, write TC codes and T*C/128 scales
    ("plain_outlier", 8192, 7168, False, 8192 * 7168 * 3 + 8192 * 56 * 4),
    # fp32 input: 4 B per element read
    ("plain_f32", 8192, 7168, False, 8192 * 7168 * 5 + 8192 * 56 * 4),
    # SwiGLU: read T*2H bf16, write T*H codes and T*H/128 scales (+ T weights)
    ("swiglu", 16384, 4096, False, 16384 * 4096 * 2 + 16384 * 2048 + 16384 * 16 * 4),
    ("swiglu_moe", 65536, 4096, True,
     65536 * 4096 * 2 + 65536 * 2048 + 65536 * 16 * 4 + 65536 * 4),
    ("swiglu_clamp", 16384, 4096, False, 16384 * 4096 * 2 + 16384 * 2048 + 16384 * 16 * 4),
    # transposed: plus H*T codes and H * T/128 scales
    ("swiglu_t", 131072, 4096, False,
     131072 * 4096 * 2 + 2 * 131072 * 2048 + 131072 * 16 * 4 + 2048 * 1024 * 4),
    ("swiglu_t_clamp", 131072, 4096, False,
     131072 * 4096 * 2 + 2 * 131072 * 2048 + 131072 * 16 * 4 + 2048 * 1024 * 4),
    # backward: read gate|up (T*2H bf16) and dy (T*H bf16), write [dg | du]
    # codes (T*2H) and scales (T*2H/128), read the weights
    ("swiglu_bwd", 65536, 4096, True,
     65536 * 4096 * 2 + 65536 * 2048 * 2 + 65536 * 4096 + 65536 * 32 * 4 + 65536 * 4),
    # per-channel: one scale per 128 tokens and channel
    ("per_channel", 16384, 7168, False, 16384 * 7168 * 3 + 128 * 7168 * 4),
    ("per_channel_t", 16384, 7168, False, 16384 * 7168 * 3 + 128 * 7168 * 4),
    # per-block: one scale per 128 x 128 block, ragged last block row
    ("per_block", 16320, 7168, False, 16320 * 7168 * 3 + 128 * 56 * 4),
    # cast back: read codes and per-token scales, write bf16
    ("cast_back", 16384, 7168, False, 16384 * 7168 * 3 + 16384 * 56 * 4),
]


@pytest.mark.parametrize("name,T,C,weighted,expected", CASES)
def test_algorithmic_bytes(name, T, C, weighted, expected):
    assert bench.algorithmic_bytes(name, T, C, weighted) == expected


def test_every_workload_has_a_byte_case():
    assert {c[0] for c in CASES} >= set(bench.KERNEL_OF) - {"plain_small"}


def test_the_headline_bytes_match_the_committed_summary():
    T, C, _ = synth.WORKLOADS["swiglu_t"]
    text = open(os.path.join(bench.ROOT, "profiles", "swiglu_cast_t_swiglu_t.md")).read()
    assert f"algorithmic_bytes_per_launch: {bench.algorithmic_bytes('swiglu_t', T, C, False)}" in text


def test_profiled_traffic_needs_the_current_sources(tmp_path, monkeypatch):
    kern, workload = "cast_back", "cast_back"
    prof = tmp_path / "profiles"
    prof.mkdir()
    csrc = tmp_path / "fp8_activation_quantization_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES[kern]:
        (csrc / f).write_text(f"// {f}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    summary = prof / f"{kern}_{workload}.md"
    summary.write_text("traffic_bytes_per_launch: 12345\n"
                       f"kernel_source_sha256: {bench.kernel_source_hash(kern)}\n")
    assert bench.profiled_traffic(kern, workload) == 12345
    (csrc / bench.KERNEL_SOURCES[kern][0]).write_text("// changed\n")
    assert bench.profiled_traffic(kern, workload) is None
    assert bench.profiled_traffic(kern, "no_such_workload") is None


def test_both_arms_describe_the_same_config():
    """The config object comes from one function for both arms; it matches the
    workload tables and the byte count."""
    for name in bench.KERNEL_OF:
        cfg = bench.workload_config(name, "e4m3", 1)
        T, C, _ = synth.WORKLOADS[bench.SYNTH_OF.get(name, name)]
        assert (cfg["T"], cfg["cols"]) == (T, C)
        assert cfg["algorithmic_bytes_per_step"] == bench.algorithmic_bytes(name, T, C,
                                                                            cfg["weighted"])
    assert bench.workload_config("swiglu_moe", "e4m3", 1)["weighted"]
    assert not bench.workload_config("swiglu_t", "e4m3", 1)["weighted"]
    assert "larger than L2" in bench.workload_config("swiglu_t", "e4m3", 1)["l2"]
    assert "rotation of buffer sets" in bench.workload_config("plain_outlier", "e4m3", 1)["l2"]
    assert "dp2" in bench.workload_config("swiglu_t", "e4m3", 2)["parallelism"]


class _Sized:
    def __init__(self, nbytes):
        self.bytes = nbytes


@pytest.mark.parametrize("nbytes,l2,expected", [
    (12_713_984, 129 << 20, 43),      # plain_small: 43 sets span >= 4 x L2
    (177_995_776, 129 << 20, 4),      # plain_outlier
    (675_545_088, 129 << 20, 2),      # larger than 4 x L2: still two sets
    (1, 129 << 20, 4 * (129 << 20)),  # degenerate tiny launch
])
def test_rotation_spans_four_times_l2(nbytes, l2, expected):
    k = bench.rotation_sets(_Sized(nbytes), l2)
    assert k == expected
    assert k >= 2 and k * nbytes >= 4 * l2
    assert (k - 1) * nbytes < 4 * l2 or k == 2


def test_bar_table_judges_the_sustained_rate():
    peak = 6759.6
    pw = {"plain_outlier/e4m3": {"sustained": {"GB/s": 6159.0}},
          "swiglu_t/e4m3": {"sustained": {"GB/s": 6964.0}},
          "swiglu/e4m3": {"sustained": {"GB/s": 5000.0}},
          "cast_back/e4m3": {"sustained": {"GB/s": 1.0}}}       # not a bar workload
    t = bench.bar_table(pw, peak)
    assert set(t) == {"plain_outlier/e4m3", "swiglu_t/e4m3", "swiglu/e4m3"}
    assert t["plain_outlier/e4m3"]["pass_measured"] and not t["plain_outlier/e4m3"]["pass_nominal"]
    assert t["swiglu_t/e4m3"]["pass_measured"] and t["swiglu_t/e4m3"]["pass_nominal"]
    assert not t["swiglu/e4m3"]["pass_measured"]   # 5000 < 0.8 x 6759.6
    assert t["swiglu_t/e4m3"]["frac_of_nominal"] == round(6964.0 / bench.NOMINAL_HBM_GBS, 4)
