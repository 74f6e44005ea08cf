"""(2) Lightning-Indexer scores (tcgen05) and (2)+(3) index-top-k on the GPU
vs the oracle.  Scores: fp32 tensor-core accumulation against float64.
Indices: bit-exact except near-ties (1e-3 of the k-th score)."""
import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_scores_close, bits, check_topk_near_tie, index_scale

pytestmark = pytest.mark.gpu


def _inputs(seed, B, Tq, N, H_I, d_I, device, per_query_w=False):
    q = S.normal_bf16(seed, 2, (B, Tq, H_I, d_I), device)
    k = S.normal_bf16(seed, 12, (B, N, d_I), device)
    if per_query_w:
        # each query's own head weights, of either sign, U(-1, 1)
        w = S.uniform_f32(seed, 9, (B, Tq, H_I), device) * 2 - 1
    else:
        w = S.uniform_f32(seed, 9, (H_I,), device)
    return q, k, w


def _case(seed, B, Tq, N, H_I, d_I, m, k, q_pos, check_rows=None, per_query_w=False):
    import long_context_sparse_23_b300 as csa
    qg, kg, wg = _inputs(seed, B, Tq, N, H_I, d_I, "cuda", per_query_w)
    qp = torch.from_numpy(np.asarray(q_pos, np.int32)).cuda()
    scores = csa.csa_index_scores(qg, kg, wg, qp, m)
    idx = csa.csa_index_topk(qg, kg, wg, qp, m, k)
    torch.cuda.synchronize()
    qc, kc, wc = _inputs(seed, B, Tq, N, H_I, d_I, "cpu", per_query_w)
    q64, k64, w64 = O.bf16_to_f64(bits(qc)), O.bf16_to_f64(bits(kc)), wc.double().numpy()
    sc = scores.cpu().numpy()
    ix = idx.cpu().numpy()
    swaps = 0
    rows = check_rows if check_rows is not None else [(b, j) for b in range(B) for j in range(Tq)]
    for b, j in rows:
        t = int(q_pos[b][j])
        wq = w64 if w64.ndim == 1 else w64[b, j]
        ref = O.indexer_scores(q64[b, j], k64[b], wq, t, m)
        n = ref.shape[0]
        assert_scores_close(sc[b, j, :n], ref, index_scale(q64[b, j], k64[b, :n], wq), f"b={b} j={j}")
        swaps += check_topk_near_tie(ix[b, j], O.topk(ref, k), ref, k, f"b={b} j={j}")
    return swaps


def test_indexer_tiny_prefill():
    """4 heads x 32 (sub-tile head count, K padded to 64 by the TMA), 64 entries."""
    _case(0, 1, 256, 64, 4, 32, 4, 16, np.arange(256)[None])


@pytest.mark.parametrize("H_I,d_I", [(8, 64), (16, 128), (32, 64), (64, 128), (128, 128)])
def test_indexer_head_shapes_ragged(H_I, d_I):
    """Ragged N (not a multiple of the 128-key tile) and a partial query group."""
    Tq = 7
    pos = np.array([[3, 100, 1999, 2000, 4003, 4010, 5000]] * 2)
    _case(5, 2, Tq, 1001, H_I, d_I, 4, 64, pos)


def test_indexer_decode_128k_full():
    """B=64 sequences, one query at 131071 each, 32768 entries, 64 heads x 128."""
    wl = S.WORKLOADS["decode_128k"]
    _case(wl.seed, wl.B, 1, wl.N, wl.H_I, wl.d_I, wl.m, wl.k, np.full((wl.B, 1), 131071))


def test_indexer_decode_1m_with_tail():
    """B=4, 262144 entries, queries at 1048572..1048575 (per-query visibility)."""
    pos = np.array([list(range((1 << 20) - 4, 1 << 20))] * 4)
    _case(4, 4, 4, 262144, 64, 128, 4, 1024, pos)


def test_indexer_prefill_8k_sampled():
    """All 8192 queries x 2048 entries on the GPU; 160 rows checked."""
    rng = np.random.default_rng(1)
    rows = [(0, int(j)) for j in np.concatenate([np.arange(12), rng.integers(0, 8192, 136), np.arange(8180, 8192)])]
    _case(1, 1, 8192, 2048, 64, 128, 4, 1024, np.arange(8192)[None], check_rows=rows)


@pytest.mark.parametrize("B,Tq,N,H_I,d_I,m,k,pos", [
    (1, 256, 64, 4, 32, 4, 16, np.arange(256)[None]),                     # 64 queries per group
    (2, 7, 1001, 64, 128, 4, 64, np.array([[3, 100, 1999, 2000, 4003, 4010, 5000]] * 2)),
    (4, 1, 32768, 64, 128, 4, 1024, np.full((4, 1), 131071)),            # decode, histogram fused
    (2, 4, 262144, 64, 128, 4, 1024, np.array([list(range((1 << 20) - 4, 1 << 20))] * 2)),
])
def test_indexer_per_query_weights(B, Tq, N, H_I, d_I, m, k, pos):
    """Per-query head weights [B, Tq, H_I] of either sign (negative scores
    included): scores against the oracle element by element, indices by the
    near-tie rule."""
    _case(7, B, Tq, N, H_I, d_I, m, k, pos, per_query_w=True)
