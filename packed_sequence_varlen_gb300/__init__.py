"""GB300 (sm_103a) packed-sequence varlen causal attention.

Python face of the C ABI in ``include/varlen_attn.h``: argument marshalling
only.  PyTorch supplies device memory and the current stream; every step of
the path (planner, metadata, tile scheduler, forward, backward) runs in the
library.  There is no CPU fallback: a missing library raises.

Layout: q [T, Hq, d], k/v [T, Hkv, d] bf16 with the last dim contiguous;
``cu_seqlens`` int32 [B+1] on the device; lse fp32 [Hq, T].
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from . import _lib
from ._lib import VarlenError, VaShape, check

__all__ = [
    "pack_next_fit", "pack_best_fit_decreasing", "build_metadata", "validate_cu_seqlens",
    "tile_sizes", "workspace_size", "plan", "varlen_attn_fwd", "varlen_attn_bwd", "varlen_attn",
    "read_status", "VarlenError", "make_shape", "library_path", "loss_targets", "token_ce",
    "IGNORE_INDEX", "unpad_index", "gather_rows", "unpad", "pad", "plan_cross", "varlen_attn_fwd_cross",
    "varlen_attn_bwd_cross",
]


def library_path() -> str:
    return _lib.LIB_PATH


def _stream(dev: torch.device | None = None):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


# ----------------------------------------------------------------- host planner

def _pack(fn, lengths, capacity: int):
    lib = _lib.load()
    src = np.asarray(lengths)
    if src.ndim != 1 or (src.size and src.dtype.kind not in "iu"):
        raise TypeError("lengths: a flat sequence of integers")
    if src.size and (src.min() < np.iinfo(np.int32).min or src.max() > np.iinfo(np.int32).max):
        raise ValueError("lengths: values must fit in int32")
    n = int(src.size)
    arr = np.zeros(max(n, 1), dtype=np.int32)
    arr[:n] = src
    order = np.empty(max(n, 1), dtype=np.int32)
    offs = np.zeros(n + 1, dtype=np.int32)
    npk = ctypes.c_int32(0)
    i32p = ctypes.POINTER(ctypes.c_int32)
    check(getattr(lib, fn)(arr.ctypes.data_as(i32p), n, int(capacity), order.ctypes.data_as(i32p),
                           offs.ctypes.data_as(i32p), ctypes.byref(npk)))
    bounds = offs[:npk.value + 1].tolist()
    flat = order[:n].tolist()
    return [flat[bounds[p]:bounds[p + 1]] for p in range(npk.value)]


def pack_next_fit(lengths, capacity: int):
    """Order-preserving next-fit; packs as lists of document indices."""
    return _pack("varlen_pack_next_fit", lengths, capacity)


def pack_best_fit_decreasing(lengths, capacity: int):
    """Best-fit-decreasing; packs as lists of document indices."""
    return _pack("varlen_pack_best_fit_decreasing", lengths, capacity)


# ----------------------------------------------------------------- metadata

def build_metadata(lengths: torch.Tensor, pad_to: int = 0, T_capacity: int | None = None):
    """Device lengths (int32) -> (cu_seqlens[n+2], position_ids[T], segment_ids[T], max_seqlen[1],
    status[1]), all int32 device tensors.  ``cu_seqlens[n+1] == cu_seqlens[n]`` means no pad."""
    assert lengths.is_cuda and lengths.dtype == torch.int32 and lengths.is_contiguous()
    n = lengths.numel()
    if T_capacity is None:
        T_capacity = max(int(pad_to), 0)
    dev = lengths.device
    cu = torch.empty(n + 2, dtype=torch.int32, device=dev)
    pos = torch.empty(max(T_capacity, 1), dtype=torch.int32, device=dev)
    seg = torch.empty(max(T_capacity, 1), dtype=torch.int32, device=dev)
    mx = torch.empty(1, dtype=torch.int32, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    check(_lib.load().varlen_build_metadata(_ptr(lengths), n, int(pad_to), int(T_capacity),
                                            _ptr(cu), _ptr(pos), _ptr(seg), _ptr(mx), _ptr(st),
                                            _stream(dev)))
    return cu, pos[:T_capacity], seg[:T_capacity], mx, st


def validate_cu_seqlens(cu_seqlens: torch.Tensor, T: int, max_seqlen: int,
                        status: torch.Tensor):
    """Enqueue the contract check; a violation sets ``status`` to VA_ERR_BAD_SEQLENS."""
    check(_lib.load().varlen_validate_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, int(T),
                                                 int(max_seqlen), _ptr(status),
                                                 _stream(cu_seqlens.device)))


def cu_seqlens_from_position_ids(position_ids: torch.Tensor, reset_at_min: bool = False,
                                 strict: bool = False):
    """Device position_ids (int32 [T]) -> (cu_seqlens[T + 1], B[1], max_seqlen[1], status[1]),
    int32 device tensors; cu_seqlens[:B + 1] is the boundary array (unwritten on error)."""
    assert position_ids.is_cuda and position_ids.dtype == torch.int32 and position_ids.is_contiguous()
    T = position_ids.numel()
    dev = position_ids.device
    cu = torch.empty(T + 1, dtype=torch.int32, device=dev)
    B = torch.empty(1, dtype=torch.int32, device=dev)
    mx = torch.empty(1, dtype=torch.int32, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    check(_lib.load().varlen_cu_seqlens_from_positions(_ptr(position_ids), T, int(reset_at_min), int(strict),
                                                       _ptr(cu), T + 1, _ptr(B), _ptr(mx), _ptr(st),
                                                       _stream(dev)))
    return cu, B, mx, st


# ----------------------------------------------------------------- shapes, plans

def make_shape(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, B: int, max_seqlen: int,
               out: torch.Tensor | None = None) -> VaShape:
    T, Hq, d = q.shape
    s = VaShape()
    s.T, s.B, s.Hq, s.Hkv, s.d, s.max_seqlen = T, B, Hq, k.shape[1], d, int(max_seqlen)
    s.q_row_stride, s.q_head_stride = q.stride(0), q.stride(1)
    s.k_row_stride, s.k_head_stride = k.stride(0), k.stride(1)
    s.v_row_stride, s.v_head_stride = v.stride(0), v.stride(1)
    o = out if out is not None else q
    s.o_row_stride, s.o_head_stride = o.stride(0), o.stride(1)
    return s


def _contig_shape(T, B, Hq, Hkv, d, max_seqlen) -> VaShape:
    s = VaShape()
    _lib.load().varlen_shape_contiguous(ctypes.byref(s), T, B, Hq, Hkv, d, int(max_seqlen))
    return s


def tile_sizes(kind: int, d: int):
    """(BM, BN) of a tile map kind: 0 forward, 1 backward kv blocks, 2 backward dQ blocks."""
    bm, bn = ctypes.c_int32(), ctypes.c_int32()
    check(_lib.load().varlen_attn_tile_sizes(kind, d, ctypes.byref(bm), ctypes.byref(bn)))
    return bm.value, bn.value


def workspace_size(T, B, Hq, Hkv, d, max_seqlen, for_bwd: bool) -> int:
    s = _contig_shape(T, B, Hq, Hkv, d, max_seqlen)
    lib = _lib.load()
    n = lib.varlen_attn_workspace_size(ctypes.byref(s), int(for_bwd))
    if n == 0:  # the shape check failed: the plan entry point reports why
        check(lib.varlen_attn_plan(ctypes.byref(s), None, 0, 1, None, 0, None, None, None))
    return n


def plan(cu_seqlens: torch.Tensor, T: int, Hq: int, Hkv: int, d: int, max_seqlen: int,
         kind: int = 0, causal: bool = True, window: int | None = None):
    """Tile map on the device: (records int32 [n, 4], n).  ``window``: causal local window
    (query i sees keys i - window .. i), None for none."""
    B = cu_seqlens.numel() - 1
    s = _contig_shape(T, B, Hq, Hkv, d, max_seqlen)
    BM, BN = tile_sizes(kind, d)
    blk = BN if kind == 1 else BM
    heads = Hkv if kind == 1 else Hq
    cap = (T // blk + B) * heads
    tm = torch.empty((max(cap, 1), 4), dtype=torch.int32, device=cu_seqlens.device)
    n = torch.zeros(1, dtype=torch.int32, device=cu_seqlens.device)
    scratch = torch.empty(B + 4, dtype=torch.int32, device=cu_seqlens.device)
    check(_lib.load().varlen_attn_plan_window(ctypes.byref(s), _ptr(cu_seqlens), kind, int(causal),
                                              -1 if window is None else int(window), _ptr(tm), cap, _ptr(n),
                                              _ptr(scratch), _stream(cu_seqlens.device)))
    k = int(n.item())
    return tm[:k], k


def read_status(ws: torch.Tensor) -> int:
    st = ctypes.c_int32(-1)
    check(_lib.load().varlen_read_status(_ptr(ws), ctypes.byref(st), _stream(ws.device)))
    return st.value


def _raise_status(ws: torch.Tensor):
    st = read_status(ws)
    if st != 0:
        raise VarlenError(st, "device-detected error (status word)")


def _check_inputs(*ts):
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("q/k/v/out tensors must be CUDA bf16 [T, H, d] with a contiguous last dim")


# ----------------------------------------------------------------- attention

def varlen_attn_fwd(q, k, v, cu_seqlens, max_seqlen: int, scale: float | None = None,
                    causal: bool = True, out=None, lse=None, workspace=None, check_status=False,
                    window: int | None = None):
    """Forward: returns (out [T,Hq,d] bf16, lse [Hq,T] fp32).  ``window``: causal local window
    (query i sees keys i - window .. i of its segment), None for none."""
    win = -1 if window is None else int(window)
    _check_inputs(q, k, v)
    T, Hq, d = q.shape
    B = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    s = make_shape(q, k, v, B, max_seqlen, out)
    lib = _lib.load()
    need = lib.varlen_attn_workspace_size(ctypes.byref(s), 0)
    if need == 0:
        check(lib.varlen_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), ctypes.byref(s),
                                         scale, int(causal), win, _ptr(out), _ptr(lse), _ptr(None), 0,
                                         _stream(q.device)))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    check(lib.varlen_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), ctypes.byref(s), scale,
                                     int(causal), win, _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel(), _stream(q.device)))
    if check_status:
        _raise_status(workspace)
    return out, lse


def varlen_attn_bwd(q, k, v, out, lse, dout, cu_seqlens, max_seqlen: int,
                    scale: float | None = None, causal: bool = True, dq=None, dk=None, dv=None,
                    workspace=None, check_status=False, window: int | None = None):
    """Backward: returns (dq, dk, dv) bf16 with the shapes of q, k, v (``window`` as in the
    forward that produced out and lse)."""
    _check_inputs(q, k, v, out, dout)
    if out.stride() != dout.stride():
        raise ValueError("out and dout must share strides")
    T, Hq, d = q.shape
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if dq is None:
        dq = torch.empty_strided(out.shape, out.stride(), dtype=q.dtype, device=q.device)
    if dk is None:
        dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    if dv is None:
        dv = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    if dq.stride() != out.stride() or dk.stride() != k.stride() or dv.stride() != k.stride():
        raise ValueError("dq must share out's strides and dk/dv k's strides")
    s = make_shape(q, k, v, B, max_seqlen, out)
    lib = _lib.load()
    need = lib.varlen_attn_workspace_size(ctypes.byref(s), 1)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(lib.varlen_attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                     _ptr(cu_seqlens), ctypes.byref(s), scale, int(causal),
                                     -1 if window is None else int(window), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(workspace), workspace.numel(), _stream(q.device)))
    if check_status:
        _raise_status(workspace)
    return dq, dk, dv


class _VarlenAttn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, max_seqlen, scale, causal, window):
        out, lse = varlen_attn_fwd(q, k, v, cu_seqlens, max_seqlen, scale, causal, window=window)
        ctx.save_for_backward(q, k, v, out, lse, cu_seqlens)
        ctx.max_seqlen, ctx.scale, ctx.causal, ctx.window = max_seqlen, scale, causal, window
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse, cu = ctx.saved_tensors
        dout = dout.contiguous() if dout.stride() != out.stride() else dout
        dq, dk, dv = varlen_attn_bwd(q, k, v, out, lse, dout, cu, ctx.max_seqlen, ctx.scale,
                                     ctx.causal, window=ctx.window)
        return dq, dk, dv, None, None, None, None, None


def varlen_attn(q, k, v, cu_seqlens, max_seqlen: int, scale: float | None = None,
                causal: bool = True, window: int | None = None):
    """Differentiable packed attention: out [T, Hq, d] (``window``: causal local window)."""
    return _VarlenAttn.apply(q, k, v, cu_seqlens, max_seqlen, scale, causal, window)


# ----------------------------------------------------------------- cross-attention

def plan_cross(cu_q: torch.Tensor, cu_k: torch.Tensor, Tq: int, Tk: int, Hq: int, Hkv: int, d: int,
               max_seqlen_q: int, kind: int = 0, causal: bool = True):
    """Cross-attention tile map on the device: (records int32 [n, 4], n)."""
    B = cu_q.numel() - 1
    s = _contig_shape(Tq, B, Hq, Hkv, d, max_seqlen_q)
    BM, BN = tile_sizes(kind, d)
    cap = ((Tk // BN) + B) * Hkv if kind == 1 else (Tq // BM + B) * Hq
    tm = torch.empty((max(cap, 1), 4), dtype=torch.int32, device=cu_q.device)
    n = torch.zeros(1, dtype=torch.int32, device=cu_q.device)
    scratch = torch.empty(B + 4, dtype=torch.int32, device=cu_q.device)
    check(_lib.load().varlen_attn_plan_cross(ctypes.byref(s), _ptr(cu_q), _ptr(cu_k), Tk, kind, int(causal),
                                             _ptr(tm), cap, _ptr(n), _ptr(scratch), _stream(cu_q.device)))
    k = int(n.item())
    return tm[:k], k


def varlen_attn_fwd_cross(q, k, v, cu_q, cu_k, max_seqlen_q: int, max_seqlen_k: int, scale: float | None = None,
                          causal: bool = True, out=None, lse=None, workspace=None, check_status=False):
    """Cross-attention forward (q [Tq,Hq,d] against k/v [Tk,Hkv,d], boundaries cu_q / cu_k;
    causal aligned bottom-right): returns (out [Tq,Hq,d] bf16, lse [Hq,Tq] fp32)."""
    _check_inputs(q, k, v)
    Tq, Hq, d = q.shape
    Tk = k.shape[0]
    B = cu_q.numel() - 1
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    s = make_shape(q, k, v, B, max_seqlen_q, out)
    lib = _lib.load()
    need = lib.varlen_attn_workspace_size_cross(ctypes.byref(s), Tk, 0)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(lib.varlen_attn_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(cu_k), ctypes.byref(s), Tk,
                                    int(max_seqlen_k), scale, int(causal), _ptr(out), _ptr(lse), _ptr(workspace),
                                    workspace.numel(), _stream(q.device)))
    if check_status:
        _raise_status(workspace)
    return out, lse


def varlen_attn_bwd_cross(q, k, v, out, lse, dout, cu_q, cu_k, max_seqlen_q: int, max_seqlen_k: int,
                          scale: float | None = None, causal: bool = True, workspace=None, check_status=False):
    """Cross-attention backward: returns (dq, dk, dv) bf16 with the shapes of q, k, v."""
    _check_inputs(q, k, v, out, dout)
    Tq, Hq, d = q.shape
    Tk = k.shape[0]
    B = cu_q.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_strided(out.shape, out.stride(), dtype=q.dtype, device=q.device)
    dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    dv = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    s = make_shape(q, k, v, B, max_seqlen_q, out)
    lib = _lib.load()
    need = lib.varlen_attn_workspace_size_cross(ctypes.byref(s), Tk, 1)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(lib.varlen_attn_bwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(cu_q),
                                    _ptr(cu_k), ctypes.byref(s), Tk, int(max_seqlen_k), scale, int(causal), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), _stream(q.device)))
    if check_status:
        _raise_status(workspace)
    return dq, dk, dv


# ----------------------------------------------------------------- packed loss

IGNORE_INDEX = -100


def loss_targets(token_ids: torch.Tensor, cu_seqlens: torch.Tensor, ignore_index: int = IGNORE_INDEX):
    """Next-token targets (int32 [T]) of a packed stream of whole documents: pairs formed
    inside each segment, ``ignore_index`` at every segment's last position."""
    if not token_ids.is_cuda or token_ids.dtype != torch.int32 or token_ids.dim() != 1:
        raise ValueError("token_ids must be a CUDA int32 [T] tensor")
    T = token_ids.numel()
    out = torch.empty(T, dtype=torch.int32, device=token_ids.device)
    check(_lib.load().varlen_loss_targets(_ptr(token_ids), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                          int(ignore_index), _ptr(out), _stream(token_ids.device)))
    return out


def token_ce(logits: torch.Tensor, targets: torch.Tensor, ignore_index: int = IGNORE_INDEX,
             grad: bool | torch.Tensor = True, workspace=None, check_status=False):
    """Token-weighted cross entropy of the packed stream: returns (loss [2] float64 device
    tensor {sum, mean}, count [1] int32, grad or None).  ``logits`` is CUDA fp32 or bf16
    [T, V] with a contiguous last dim; ``grad`` True allocates d(mean)/d(logits) like
    ``logits``, a tensor receives it, False skips it."""
    if not logits.is_cuda or logits.dim() != 2 or logits.stride(1) != 1 or \
            logits.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("logits must be a CUDA fp32/bf16 [T, V] tensor with a contiguous last dim")
    T, V = logits.shape
    dev = logits.device
    if grad is True:
        g = torch.empty_like(logits, memory_format=torch.contiguous_format)
    elif grad is False or grad is None:
        g = None
    else:
        g = grad
        if g.shape != logits.shape or g.dtype != logits.dtype or g.stride(1) != 1:
            raise ValueError("grad must match logits in shape and dtype, with a contiguous last dim")
    lib = _lib.load()
    need = lib.varlen_token_ce_workspace_size(T)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    loss = torch.empty(2, dtype=torch.float64, device=dev)
    count = torch.empty(1, dtype=torch.int32, device=dev)
    check(lib.varlen_token_ce(_ptr(logits), 1 if logits.dtype == torch.bfloat16 else 0, logits.stride(0),
                              _ptr(targets), T, V, int(ignore_index), _ptr(loss), _ptr(count), _ptr(g),
                              g.stride(0) if g is not None else 0, _ptr(workspace), workspace.numel(),
                              _stream(dev)))
    if check_status:
        _raise_status(workspace)
    return loss, count, g


# ----------------------------------------------------------------- padded-batch bridge

def unpad_index(mask: torch.Tensor):
    """Padded batch -> packed stream.  ``mask`` CUDA [Bp, S] (nonzero = real token).  Returns
    (indices [Bp*S], inverse [Bp*S], cu_seqlens [Bp+1] (int32 device tensors), T, max_seqlen);
    T and max_seqlen are read back to the host (one synchronisation), as the attention calls
    take them on the host.  A row without real tokens raises (status VA_ERR_BAD_SEQLENS)."""
    if not mask.is_cuda or mask.dim() != 2:
        raise ValueError("mask must be a CUDA [Bp, S] tensor")
    m = mask.to(torch.int32).contiguous()
    Bp, S = m.shape
    dev = m.device
    indices = torch.empty(Bp * S, dtype=torch.int32, device=dev)
    inverse = torch.empty(Bp * S, dtype=torch.int32, device=dev)
    cu = torch.empty(Bp + 1, dtype=torch.int32, device=dev)
    small = torch.empty(3, dtype=torch.int32, device=dev)  # T, max_seqlen, status
    check(_lib.load().varlen_unpad_index(_ptr(m), Bp, S, _ptr(indices), _ptr(inverse), _ptr(cu),
                                         ctypes.c_void_p(small.data_ptr()),
                                         ctypes.c_void_p(small.data_ptr() + 4),
                                         ctypes.c_void_p(small.data_ptr() + 8), _stream(dev)))
    T, mx, st = (int(x) for x in small.cpu())
    if st != 0:
        raise VarlenError(st, "unpad_index: a row has no real token")
    return indices, inverse, cu, T, mx


def gather_rows(src: torch.Tensor, row_map: torch.Tensor, n_rows: int) -> torch.Tensor:
    """dst[i] = src[row_map[i]] (a zero row where row_map[i] < 0) for i < n_rows; rows are
    src's trailing dims (contiguous, a multiple of 16 bytes)."""
    if not src.is_cuda or src.dim() < 1 or not src[0].is_contiguous():
        raise ValueError("src must be a CUDA tensor with contiguous rows")
    row_bytes = src[0].numel() * src.element_size()
    dst = torch.empty((n_rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    check(_lib.load().varlen_gather_rows(_ptr(src), src.stride(0) * src.element_size(), _ptr(row_map), n_rows,
                                         row_bytes, _ptr(dst), dst.stride(0) * dst.element_size(),
                                         _stream(src.device)))
    return dst


def unpad(x: torch.Tensor, indices: torch.Tensor, T: int) -> torch.Tensor:
    """[Bp, S, ...] -> [T, ...]: the real tokens in row-major order."""
    return gather_rows(x.reshape((-1,) + tuple(x.shape[2:])), indices, T)


def pad(y: torch.Tensor, inverse: torch.Tensor, Bp: int, S: int) -> torch.Tensor:
    """[T, ...] -> [Bp, S, ...]: each token back to its padded position, zeros in the padding."""
    return gather_rows(y, inverse, Bp * S).reshape((Bp, S) + tuple(y.shape[1:]))
