"""Host-side bookkeeping of bench.py on the CPU: the kernel launches claimed per
decode step follow the library's launch plan for each workload."""
import os
import sys
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import csa_synth as S  # noqa: E402


def _launches(name, Tq=None):
    wl = S.WORKLOADS[name]
    ds = SimpleNamespace(wl=wl, Tq=Tq if Tq is not None else len(wl.q_positions))
    return bench.DecodeStep.kernels_per_step(ds)


def test_decode_1m_step_is_zeroing_indexer_and_fused_tail():
    assert _launches("decode_1m") == 3


def test_decode_128k_step_is_one_pass_topk_and_cluster_merged_attention():
    # 32768 entries: one top-k kernel; 1024 + 128 slots = 9 tiles -> 2 ranges,
    # merged inside their cluster (no merge kernel)
    assert _launches("decode_128k") == 2 + 1 + 1


def test_mid_and_long_rows_and_many_ranges():
    wl = S.WORKLOADS["decode_128k"]
    count = lambda **kw: bench.DecodeStep.kernels_per_step(SimpleNamespace(wl=wl.replace(**kw), Tq=1))
    assert count(T=4 * 40000) == 2 + 2 + 1              # select + finish between 32768 and 65536 entries
    assert count(T=4 * 16384) == 2 + 1                  # short rows: indexer, one-pass top-k, attention
    assert count(T=4 * 40000, k=4096) == 2 + 2 + 1      # 33 tiles -> 7 ranges: merged in the cluster
    assert count(T=4 * 40000, k=5200) == 2 + 2 + 1 + 1  # 42 tiles -> 9 ranges: the merge kernel too


def test_tail_queries_need_the_histogram_pass():
    assert _launches("decode_1m_tail") == 4
