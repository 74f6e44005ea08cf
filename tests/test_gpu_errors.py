"""Device-side failure reporting without faulting the GPU: a bounded wait that
runs out sets CSA_FLAG_TIMEOUT in the workspace error word and the kernel
returns; the context stays usable and the next call is correct."""
import numpy as np
import pytest
import torch

import csa_synth as S
from long_context_sparse_23_b300 import _lib

pytestmark = pytest.mark.gpu


def test_wait_budget_runs_out_and_context_survives():
    import long_context_sparse_23_b300 as csa
    q = S.normal_bf16(1, 2, (2, 1, 64, 128), "cuda")
    k = S.normal_bf16(1, 12, (2, 4096, 128), "cuda")
    w = S.uniform_f32(1, 9, (64,), "cuda")
    qp = torch.tensor([[16383], [16383]], dtype=torch.int32, device="cuda")
    ws = csa.Workspace()
    ref = csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
    assert ws.check_error() == 0
    try:
        _lib.lib().csa_set_wait_budget(1)       # one clock cycle: the first real wait gives up
        csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
        flags = ws.check_error()
    finally:
        _lib.lib().csa_set_wait_budget(0)       # back to the default budget
    assert flags & _lib.CSA_FLAG_TIMEOUT
    again = csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
    assert ws.check_error() == 0
    assert torch.equal(again, ref)
