"""B300 (sm_103a) Compressed Sparse Attention: Python binding of libcsa.so.

The functions here carry the C ABI's names and only marshal arguments: every
step of the path runs in the library's CUDA kernels, on the current torch
stream.  Tensors must be CUDA, contiguous, bf16 where the C ABI says bf16,
int32 for positions and indices, fp32 for the indexer weights.

    csa_compress     (1) block compression of up to three streams
    csa_append       (1') decode-time compression of completed blocks into the caches
    csa_index_scores (2) Lightning-Indexer scores
    csa_topk         (3) per-query top-k of given scores
    csa_index_topk   (2)+(3)
    csa_quantize_fp8, csa_index_scores_fp8   (2') the indexer on E4M3 rows
    csa_attend       (4) attention over selected entries + sliding window
    hca_attend       dense HCA mode + sliding window
    csa_layer        (1)->(4) in one call
"""
from __future__ import annotations

import ctypes
import math
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import CSA_BF16, CSA_F32, CsaError, check, csa_layer_args

__all__ = ["csa_compress", "csa_append", "csa_index_scores", "csa_topk", "csa_index_topk", "csa_attend",
           "hca_attend", "csa_layer", "Workspace", "CsaError", "scores_ld"]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _odt(dtype) -> int:
    if dtype == torch.bfloat16:
        return CSA_BF16
    if dtype == torch.float32:
        return CSA_F32
    raise ValueError("out dtype must be torch.bfloat16 or torch.float32")


def scores_ld(N: int) -> int:
    return (N + 3) // 4 * 4


class Workspace:
    """Device scratch for the library calls (error word + temporaries).

    One workspace per stream; calls that overlap on the GPU must not share it.
    """

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.buf = None
        self.nbytes = 0
        self.ensure(max(nbytes, _lib.CSA_WS_HEADER_BYTES))

    def ensure(self, nbytes: int) -> "Workspace":
        if nbytes > self.nbytes:
            self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
            self.nbytes = nbytes
            check("csa_workspace_init", _lib.lib().csa_workspace_init(self.ptr, self.nbytes, _stream()))
        return self

    @property
    def ptr(self) -> int:
        p = self.buf.data_ptr()
        return (p + 255) // 256 * 256

    def check_error(self, clear: bool = True) -> int:
        """Synchronise the stream and return the device error bits (0 = none)."""
        flags = ctypes.c_uint32(0)
        st = _lib.lib().csa_check_error(self.ptr, ctypes.byref(flags), int(clear), _stream())
        if st not in (_lib.CSA_OK, _lib.CSA_ERR_TIMEOUT, _lib.CSA_ERR_DEVICE_INDEX):
            check("csa_check_error", st)
        return flags.value


_ws_cache: Dict[Tuple[int, int], Workspace] = {}


def _ws(nbytes: int, ws: Optional[Workspace]) -> Workspace:
    if ws is not None:
        return ws.ensure(nbytes)
    key = (torch.cuda.current_device(), _stream())
    w = _ws_cache.get(key)
    if w is None:
        w = _ws_cache[key] = Workspace(nbytes)
    return w.ensure(nbytes)


def default_workspace() -> Workspace:
    return _ws(_lib.CSA_WS_HEADER_BYTES, None)


# ---------------------------------------------------------------- (1)

def csa_compress(xs: Sequence[torch.Tensor], gs: Sequence[torch.Tensor], m: int,
                 out_dtype=torch.bfloat16, outs: Optional[Sequence[torch.Tensor]] = None) -> List[torch.Tensor]:
    n = len(xs)
    B, T = xs[0].shape[0], xs[0].shape[1]
    if outs is None:
        outs = [torch.empty(B, T // m, x.shape[2], dtype=out_dtype, device=x.device) for x in xs]
    P = ctypes.c_void_p * 3
    D = (ctypes.c_int * 3)(*[x.shape[2] for x in xs] + [0] * (3 - n))
    st = _lib.lib().csa_compress(n, P(*[_ptr(x) for x in xs]), P(*[_ptr(g) for g in gs]),
                                 P(*[_ptr(o) for o in outs]), D, B, T, m, _odt(outs[0].dtype), _stream())
    check("csa_compress", st)
    return list(outs)


def csa_append(x_wins: Sequence[torch.Tensor], g_wins: Sequence[torch.Tensor], outs: Sequence[torch.Tensor],
               raw_base: torch.Tensor, q_pos: torch.Tensor, m: int, ws: Optional[Workspace] = None) -> None:
    """Decode-time compression: the blocks completed by the positions q_pos,
    from the window rows x_wins / g_wins ([B, T_raw, D]) into the caches outs
    ([B, N, D] bf16), in place."""
    n = len(x_wins)
    B, T_raw = x_wins[0].shape[0], x_wins[0].shape[1]
    P = ctypes.c_void_p * 3
    D = (ctypes.c_int * 3)(*[x.shape[2] for x in x_wins] + [0] * (3 - n))
    w_ = _ws(_lib.CSA_WS_HEADER_BYTES, ws)
    st = _lib.lib().csa_append(n, P(*[_ptr(x) for x in x_wins]), P(*[_ptr(g) for g in g_wins]),
                               P(*[_ptr(o) for o in outs]), D, _ptr(raw_base), _ptr(q_pos), B, q_pos.shape[1],
                               T_raw, outs[0].shape[1], m, w_.ptr, w_.nbytes, _stream())
    check("csa_append", st)


# ---------------------------------------------------------------- (2), (3)

def _w_stride(w: torch.Tensor, B: int, Tq: int, H_I: int) -> int:
    """0 for one [H_I] weight vector shared by every query; H_I for per-query
    weights [B, Tq, H_I]."""
    if w.dim() == 1:
        return 0
    if tuple(w.shape) != (B, Tq, H_I):
        raise ValueError("indexer weights must be [H_I] or [B, Tq, H_I]")
    return H_I


def csa_index_scores(q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor, q_pos: torch.Tensor,
                     m: int, scores: Optional[torch.Tensor] = None,
                     ws: Optional[Workspace] = None) -> torch.Tensor:
    B, Tq, H_I, d_I = q_idx.shape
    N = k_idx.shape[1]
    if scores is None:
        scores = torch.full((B, Tq, scores_ld(N)), float("nan"), dtype=torch.float32, device=q_idx.device)
    w_ = _ws(_lib.CSA_WS_HEADER_BYTES, ws)
    st = _lib.lib().csa_index_scores(_ptr(q_idx), _ptr(k_idx), _ptr(w), _w_stride(w, B, Tq, H_I), _ptr(q_pos),
                                     B, Tq, N, H_I, d_I, m,
                                     _ptr(scores), scores.shape[-1], w_.ptr, w_.nbytes, _stream())
    check("csa_index_scores", st)
    return scores


def csa_quantize_fp8(x: torch.Tensor):
    """Rows of x (bf16, last dimension D) -> (E4M3 codes as uint8, same shape;
    fp32 power-of-two scale per row, shape x.shape[:-1])."""
    D = x.shape[-1]
    rows = x.numel() // D
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    check("csa_quantize_fp8", _lib.lib().csa_quantize_fp8(_ptr(x), rows, D, _ptr(codes), _ptr(scales), _stream()))
    return codes, scales


def csa_index_scores_fp8(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor, k_scale: torch.Tensor,
                         w: torch.Tensor, q_pos: torch.Tensor, m: int, scores: Optional[torch.Tensor] = None,
                         ws: Optional[Workspace] = None) -> torch.Tensor:
    """(2) on E4M3 rows: q8 [B, Tq, H_I, d_I] / q_scale [B, Tq, H_I] and
    k8 [B, N, d_I] / k_scale [B, N] as made by csa_quantize_fp8."""
    B, Tq, H_I, d_I = q8.shape
    N = k8.shape[1]
    if scores is None:
        scores = torch.full((B, Tq, scores_ld(N)), float("nan"), dtype=torch.float32, device=q8.device)
    w_ = _ws(_lib.CSA_WS_HEADER_BYTES, ws)
    st = _lib.lib().csa_index_scores_fp8(_ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(w),
                                         _w_stride(w, B, Tq, H_I), _ptr(q_pos), B, Tq, N, H_I, d_I, m,
                                         _ptr(scores), scores.shape[-1], w_.ptr, w_.nbytes, _stream())
    check("csa_index_scores_fp8", st)
    return scores


def csa_topk(scores: torch.Tensor, q_pos: torch.Tensor, N: int, m: int, k: int,
             with_scores: bool = False, ws: Optional[Workspace] = None):
    B, Tq, ld = scores.shape
    idx = torch.empty(B, Tq, k, dtype=torch.int32, device=scores.device)
    sel = torch.empty(B, Tq, k, dtype=torch.float32, device=scores.device) if with_scores else None
    need = ctypes.c_size_t(0)
    check("csa_topk_workspace", _lib.lib().csa_topk_workspace(B, Tq, N, k, ctypes.byref(need)))
    w_ = _ws(need.value, ws)
    st = _lib.lib().csa_topk(_ptr(scores), ld, _ptr(q_pos), B, Tq, N, m, k, _ptr(idx), _ptr(sel),
                             w_.ptr, w_.nbytes, _stream())
    check("csa_topk", st)
    return (idx, sel) if with_scores else idx


def csa_index_topk(q_idx: torch.Tensor, k_idx: torch.Tensor, w: torch.Tensor, q_pos: torch.Tensor,
                   m: int, k: int, with_scores: bool = False, ws: Optional[Workspace] = None):
    B, Tq, H_I, d_I = q_idx.shape
    N = k_idx.shape[1]
    need = ctypes.c_size_t(0)
    check("csa_index_topk_workspace",
          _lib.lib().csa_index_topk_workspace(B, Tq, N, H_I, d_I, k, ctypes.byref(need)))
    w_ = _ws(need.value, ws)
    idx = torch.empty(B, Tq, k, dtype=torch.int32, device=q_idx.device)
    sel = torch.empty(B, Tq, k, dtype=torch.float32, device=q_idx.device) if with_scores else None
    st = _lib.lib().csa_index_topk(_ptr(q_idx), _ptr(k_idx), _ptr(w), _w_stride(w, B, Tq, H_I), _ptr(q_pos),
                                   B, Tq, N, H_I, d_I, m, k,
                                   _ptr(idx), _ptr(sel), w_.ptr, w_.nbytes, _stream())
    check("csa_index_topk", st)
    return (idx, sel) if with_scores else idx


# ---------------------------------------------------------------- (4)

def csa_attend(q, k_cmp, v_cmp, idx, k_raw, v_raw, raw_base, q_pos, W: int, scale: float = 0.0,
               out_dtype=torch.bfloat16, with_lse: bool = False, ws: Optional[Workspace] = None):
    B, Tq, H, d = q.shape
    N = k_cmp.shape[1]
    T_raw = k_raw.shape[1] if k_raw is not None else 0
    k = idx.shape[-1]
    need = ctypes.c_size_t(0)
    check("csa_attend_workspace", _lib.lib().csa_attend_workspace(B, Tq, H, d, k, W, ctypes.byref(need)))
    w_ = _ws(need.value, ws)
    out = torch.empty(B, Tq, H, d, dtype=out_dtype, device=q.device)
    lse = torch.empty(B, Tq, H, dtype=torch.float32, device=q.device) if with_lse else None
    st = _lib.lib().csa_attend(_ptr(q), _ptr(k_cmp), _ptr(v_cmp), _ptr(idx), _ptr(k_raw), _ptr(v_raw),
                               _ptr(raw_base), _ptr(q_pos), B, Tq, N, T_raw, H, d, k, W, float(scale),
                               _ptr(out), _odt(out_dtype), _ptr(lse), w_.ptr, w_.nbytes, _stream())
    check("csa_attend", st)
    return (out, lse) if with_lse else out


def hca_attend(q, k_cmp, v_cmp, k_raw, v_raw, raw_base, q_pos, m: int, W: int, scale: float = 0.0,
               out_dtype=torch.bfloat16, with_lse: bool = False, ws: Optional[Workspace] = None):
    B, Tq, H, d = q.shape
    N = k_cmp.shape[1]
    T_raw = k_raw.shape[1] if k_raw is not None else 0
    need = ctypes.c_size_t(0)
    check("hca_attend_workspace", _lib.lib().hca_attend_workspace(B, Tq, N, H, d, W, ctypes.byref(need)))
    w_ = _ws(need.value, ws)
    out = torch.empty(B, Tq, H, d, dtype=out_dtype, device=q.device)
    lse = torch.empty(B, Tq, H, dtype=torch.float32, device=q.device) if with_lse else None
    st = _lib.lib().hca_attend(_ptr(q), _ptr(k_cmp), _ptr(v_cmp), _ptr(k_raw), _ptr(v_raw), _ptr(raw_base),
                               _ptr(q_pos), B, Tq, N, T_raw, H, d, m, W, float(scale), _ptr(out),
                               _odt(out_dtype), _ptr(lse), w_.ptr, w_.nbytes, _stream())
    check("hca_attend", st)
    return (out, lse) if with_lse else out


# ---------------------------------------------------------------- layer

def layer_args(*, B, Tq, N, m, H, d, H_I, d_I, k, W, T=0, T_raw=0, scale=0.0, x_k=None, x_v=None, x_i=None,
               g_k=None, g_v=None, g_i=None, k_cmp=None, v_cmp=None, i_cmp=None, k_win=None, v_win=None,
               raw_base=None, q=None, q_idx=None, w=None, q_pos=None, idx_out=None, out=None,
               out_dtype=torch.bfloat16, lse=None, i_win=None, gk_win=None, gv_win=None,
               gi_win=None, i_scale=None) -> csa_layer_args:
    a = csa_layer_args()
    for name, v in dict(B=B, Tq=Tq, N=N, m=m, H=H, d=d, H_I=H_I, d_I=d_I, k=k, W=W, T=T, T_raw=T_raw).items():
        setattr(a, name, int(v))
    a.scale = float(scale)
    for name, t in dict(x_k=x_k, x_v=x_v, x_i=x_i, g_k=g_k, g_v=g_v, g_i=g_i, k_cmp=k_cmp, v_cmp=v_cmp,
                        i_cmp=i_cmp, k_win=k_win, v_win=v_win, raw_base=raw_base, q=q, q_idx=q_idx, w=w,
                        q_pos=q_pos, idx_out=idx_out, out=out, lse=lse, i_win=i_win, gk_win=gk_win,
                        gv_win=gv_win, gi_win=gi_win, i_scale=i_scale).items():
        setattr(a, name, _ptr(t))
    a.out_dtype = _odt(out_dtype)
    a.w_stride = 0 if w is None or w.dim() == 1 else int(w.shape[-1])
    return a


def csa_layer(args: csa_layer_args, ws: Optional[Workspace] = None) -> None:
    need = ctypes.c_size_t(0)
    check("csa_layer_workspace", _lib.lib().csa_layer_workspace(ctypes.byref(args), ctypes.byref(need)))
    w_ = _ws(need.value, ws)
    check("csa_layer", _lib.lib().csa_layer(ctypes.byref(args), w_.ptr, w_.nbytes, _stream()))


def csa_layer_prefill(inp: Dict[str, torch.Tensor], m: int, k: int, W: int, scale: float = 0.0,
                      out_dtype=torch.bfloat16, ws: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    """Steps (1)-(4) for a prefill: every raw token is a query and the raw
    streams double as the window buffer.  Returns the caches, indices and output."""
    q, q_idx = inp["q"], inp["q_idx"]
    B, T, H, d = q.shape
    H_I, d_I = q_idx.shape[2], q_idx.shape[3]
    N = T // m
    dev = q.device
    k_cmp = torch.empty(B, N, d, dtype=torch.bfloat16, device=dev)
    v_cmp = torch.empty(B, N, d, dtype=torch.bfloat16, device=dev)
    i_cmp = torch.empty(B, N, d_I, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(B, T, k, dtype=torch.int32, device=dev)
    out = torch.empty(B, T, H, d, dtype=out_dtype, device=dev)
    a = layer_args(B=B, Tq=T, N=N, m=m, H=H, d=d, H_I=H_I, d_I=d_I, k=k, W=W, T=T, T_raw=T, scale=scale,
                   x_k=inp["k_raw"], x_v=inp["v_raw"], x_i=inp["i_raw"], g_k=inp["g_k"], g_v=inp["g_v"],
                   g_i=inp["g_i"], k_cmp=k_cmp, v_cmp=v_cmp, i_cmp=i_cmp, k_win=inp["k_raw"],
                   v_win=inp["v_raw"], raw_base=inp["raw_base"], q=q, q_idx=q_idx, w=inp["w"],
                   q_pos=inp["q_pos"], idx_out=idx, out=out, out_dtype=out_dtype)
    csa_layer(a, ws)
    return {"k_cmp": k_cmp, "v_cmp": v_cmp, "i_cmp": i_cmp, "idx": idx, "out": out}
