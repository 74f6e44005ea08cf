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


def test_decode_128k_step_adds_select_finish_attention_and_range_merge():
    # 1024 + 128 slots = 9 tiles -> 3 ranges -> the merge kernel runs too
    assert _launches("decode_128k") == 2 + 2 + 2


def test_tail_queries_need_the_histogram_pass():
    assert _launches("decode_1m_tail") == 4
