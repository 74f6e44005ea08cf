"""The hybrid layer stack at decode time (two sliding-window layers, then
CSA and HCA alternating; each layer's output is the next layer's query and
indexer query) on the GPU.  The stack is run on its prefixes of 1 .. L
layers, so every layer is checked against the oracle on the GPU's own input
activation for that layer: CSA indices by the near-tie rule, outputs within
1e-2 + 1e-2 |ref|."""
import ctypes
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from long_context_sparse_23_b300 import _lib
from tests._parity import assert_attention_close, bits, check_topk_near_tie

pytestmark = pytest.mark.gpu

KINDS = [_lib.CSA_STACK_SWA, _lib.CSA_STACK_SWA, _lib.CSA_STACK_CSA, _lib.CSA_STACK_HCA,
         _lib.CSA_STACK_CSA, _lib.CSA_STACK_HCA]


def test_stack_layer_by_layer():
    import long_context_sparse_23_b300 as csa
    B, H, d, H_I, d_I, m, m_h, k, W, T_raw = 2, 64, 128, 64, 128, 4, 128, 256, 128, 256
    t = 4095
    N, N_h = (t + 1) // m, (t + 1) // m_h
    dev = "cuda"
    q_pos = torch.full((B, 1), t, dtype=torch.int32, device=dev)
    raw_base = torch.full((B,), t + 1 - T_raw, dtype=torch.int32, device=dev)
    layers = (_lib.csa_stack_layer * len(KINDS))()
    keep, tensors = [], []
    for i, kind in enumerate(KINDS):
        seed = 60 + i
        kw = S.normal_bf16(seed, S.TID["k_raw"], (B, T_raw, d), dev)
        vw = S.normal_bf16(seed, S.TID["v_raw"], (B, T_raw, d), dev)
        L = dict(kind=kind, k_win=kw, v_win=vw)
        if kind == _lib.CSA_STACK_CSA:
            L.update(k_cmp=S.normal_bf16(seed, S.TID["k_cmp"], (B, N, d), dev),
                     v_cmp=S.normal_bf16(seed, S.TID["v_cmp"], (B, N, d), dev),
                     i_cmp=S.normal_bf16(seed, S.TID["i_cmp"], (B, N, d_I), dev),
                     w=S.uniform_f32(seed, S.TID["w"], (H_I,), dev),
                     idx=torch.empty(B, 1, k, dtype=torch.int32, device=dev))
            a = csa.layer_args(B=B, Tq=1, N=N, m=m, H=H, d=d, H_I=H_I, d_I=d_I, k=k, W=W, T_raw=T_raw,
                               k_cmp=L["k_cmp"], v_cmp=L["v_cmp"], i_cmp=L["i_cmp"], k_win=kw, v_win=vw,
                               raw_base=raw_base, w=L["w"], q_pos=q_pos, idx_out=L["idx"])
        elif kind == _lib.CSA_STACK_HCA:
            L.update(k_cmp=S.normal_bf16(seed, S.TID["k_cmp"], (B, N_h, d), dev),
                     v_cmp=S.normal_bf16(seed, S.TID["v_cmp"], (B, N_h, d), dev))
            a = csa.layer_args(B=B, Tq=1, N=N_h, m=m_h, H=H, d=d, H_I=0, d_I=0, k=0, W=W, T_raw=T_raw,
                               k_cmp=L["k_cmp"], v_cmp=L["v_cmp"], k_win=kw, v_win=vw, raw_base=raw_base,
                               q_pos=q_pos)
        else:
            a = csa.layer_args(B=B, Tq=1, N=0, m=1, H=H, d=d, H_I=0, d_I=0, k=0, W=W, T_raw=T_raw, k_win=kw,
                               v_win=vw, raw_base=raw_base, q_pos=q_pos)
        layers[i].kind = kind
        layers[i].a = a
        tensors.append(L)
    x = S.normal_bf16(59, S.TID["q"], (B, 1, H, d), dev)
    Lib = _lib.lib()
    st = torch.cuda.current_stream().cuda_stream
    acts = [x]
    for n in range(1, len(KINDS) + 1):
        need = ctypes.c_size_t(0)
        assert Lib.csa_stack_workspace(layers, n, ctypes.byref(need)) == 0
        ws = csa.Workspace(need.value)
        y = torch.empty(B, 1, H, d, dtype=torch.bfloat16, device=dev)
        r = Lib.csa_stack_decode(layers, n, x.data_ptr(), y.data_ptr(), _lib.CSA_BF16, ws.ptr, ws.nbytes, st)
        assert r == 0, Lib.csa_status_string(r)
        assert ws.check_error() == 0
        acts.append(y)
    scale = 1 / math.sqrt(d)
    rb = int(raw_base[0])
    for i, kind in enumerate(KINDS):
        L = tensors[i]
        xin = O.bf16_to_f64(bits(acts[i]))          # the GPU's input activation of layer i
        got = O.bf16_to_f64(bits(acts[i + 1]))
        kw, vw = O.bf16_to_f64(bits(L["k_win"])), O.bf16_to_f64(bits(L["v_win"]))
        win = O.window_rows(t, W, rb, T_raw)
        for b in range(B):
            if kind == _lib.CSA_STACK_SWA:
                o, _ = O.attend_one(xin[b, 0], np.zeros((0, d)), np.zeros((0, d)), [], kw[b], vw[b], win, scale)
            elif kind == _lib.CSA_STACK_HCA:
                o, _ = O.attend_one(xin[b, 0], O.bf16_to_f64(bits(L["k_cmp"]))[b], O.bf16_to_f64(bits(L["v_cmp"]))[b],
                                    np.arange(O.n_visible(t, m_h, N_h)), kw[b], vw[b], win, scale)
            else:
                S_ref = O.indexer_scores(xin[b, 0].reshape(H_I, d_I), O.bf16_to_f64(bits(L["i_cmp"]))[b],
                                         L["w"].cpu().double().numpy(), t, m)
                gidx = L["idx"][b, 0].cpu().numpy()
                check_topk_near_tie(gidx, O.topk(S_ref, k), S_ref, k, f"layer {i} b={b}")
                o, _ = O.attend_one(xin[b, 0], O.bf16_to_f64(bits(L["k_cmp"]))[b], O.bf16_to_f64(bits(L["v_cmp"]))[b],
                                    gidx, kw[b], vw[b], win, scale)
            assert_attention_close(got[b, 0], o, f"layer {i} ({kind}) b={b}")
