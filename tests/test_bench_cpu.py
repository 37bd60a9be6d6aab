"""CPU checks of bench.py's bookkeeping: the source hashes that key the
recorded DRAM traffic, the table's kernel names, and the whole-oracle timer."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_source_hash_of_one_file_and_of_a_list():
    assert bench._src_hash("bwd_bf16.cu") == bench._src_hash(("bwd_bf16.cu",))
    assert bench._src_hash(("fwd_bf16.cu", "fwd_softmax.cuh")) != bench._src_hash("fwd_bf16.cu")
    assert len(bench._src_hash("ffn.cu")) == 64


def test_traffic_table_names_known_kernels():
    from ring_attention_fwd_gb300 import binding
    known = set(binding.KERNEL_NAMES.values()) | {"ffn_up", "ffn_down"}
    for name, rec in bench.NCU_TRAFFIC.items():
        assert name in known, name
        assert len(rec["sha256"]) == 64 and rec["bytes_per_launch"] > 0


def test_oracle_full_times_every_head():
    from ring_attention_fwd_gb300.inputs import make_inputs
    inp = make_inputs(1, 2, 64, 16, 5, with_grad=True)
    w = dict(N=4, causal=True, layout="striped")
    f, t, desc = bench.oracle_full(inp, w, True)
    f1, _, _ = bench.oracle_full(inp, w, False)
    assert t > 0 and f == pytest.approx(3.5 * f1) and "2 heads" in desc
