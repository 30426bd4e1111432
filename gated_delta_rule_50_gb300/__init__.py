"""GB300 (sm_103a) gated delta rule chunked prefill -- Python binding.

Thin ctypes marshalling onto the C ABI in ``include/gdn.h`` (``libgdn.so``).
Every step of the operator runs in this package's CUDA kernels; PyTorch only
provides device memory (outputs and the workspace) and the current stream.
There is no CPU or library fallback: if the CUDA library cannot be built or
loaded, or a tensor is not on a CUDA device, the call raises.

API (flash_qla 0.1.2 README, "Usage / High-level API" and "Low-level API"):

    o, final_state = chunk_gated_delta_rule(q, k, v, g, beta, scale=None,
        initial_state=None, output_final_state=False, cu_seqlens=None)
    g_cum, A, o, h, final_state = chunk_gated_delta_rule_fwd(q, k, v, g, beta,
        scale=None, initial_state=None, cu_seqlens=None)
    dq, dk, dv, db, dg, dh0 = chunk_gated_delta_rule_bwd(q, k, v, g_cum, beta,
        A, do, dht=None, scale=None, initial_state=None, cu_seqlens=None)

plus the save-for-backward pair that training through ``chunk_gated_delta_rule`` uses (the forward
keeps its operand images and chunk-entry states; the backward skips its recompute passes):

    g_cum, A, o, final_state, saved = chunk_gated_delta_rule_fwd_saved(q, k, v, g, beta, ...)
    dq, dk, dv, db, dg, dh0 = chunk_gated_delta_rule_bwd_saved(q, k, v, g_cum, beta, A, do, saved, ...)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = ["chunk_gated_delta_rule", "chunk_gated_delta_rule_fwd", "chunk_gated_delta_rule_bwd",
           "chunk_gated_delta_rule_fwd_saved", "chunk_gated_delta_rule_bwd_saved", "SavedForward",
           "cp_plan", "cp_trigger", "GdnError", "load_library", "library_path", "workspace_bytes", "CHUNK"]

CHUNK = 64
GDN_F32, GDN_BF16 = 0, 1
CP_MODES = {"auto": 0, "off": 1, "warmup": 2}
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported problem",
           3: "workspace too small or misaligned", 4: "CUDA error", 5: "device-side wait timed out",
           6: "problem exceeds the fixed no-alloc scratch"}


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(status, status)} (gdn status {status})")
        self.status = status


class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("Hq", ctypes.c_int64),
                ("Hv", ctypes.c_int64), ("K", ctypes.c_int64), ("V", ctypes.c_int64),
                ("n_seqs", ctypes.c_int64), ("cu_seqlens", ctypes.c_void_p),
                ("cu_seqlens_host", ctypes.c_void_p), ("io_dtype", ctypes.c_int),
                ("scale", ctypes.c_float), ("cp_mode", ctypes.c_int32),
                ("warmup_chunks", ctypes.c_int32), ("out_f32", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load_library():
    """Builds (if needed) and loads libgdn.so; raises if either fails."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            P, SZ = ctypes.c_void_p, ctypes.c_size_t
            pp = ctypes.POINTER(_Problem)
            lib.gdn_fwd_workspace_bytes.argtypes = [pp]
            lib.gdn_fwd_workspace_bytes.restype = SZ
            lib.gdn_bwd_workspace_bytes.argtypes = [pp]
            lib.gdn_bwd_workspace_bytes.restype = SZ
            lib.gdn_fwd.argtypes = [pp] + [P] * 11 + [P, SZ, P]
            lib.gdn_fwd.restype = ctypes.c_int
            lib.gdn_bwd.argtypes = [pp] + [P] * 15 + [P, SZ, P]
            lib.gdn_bwd.restype = ctypes.c_int
            lib.gdn_bwd_saved_workspace_bytes.argtypes = [pp]
            lib.gdn_bwd_saved_workspace_bytes.restype = SZ
            lib.gdn_bwd_saved_uses_saved.argtypes = [pp]
            lib.gdn_bwd_saved_uses_saved.restype = ctypes.c_int
            lib.gdn_bwd_saved.argtypes = [pp] + [P] * 10 + [P, SZ] + [P] * 6 + [P, SZ, P]
            lib.gdn_bwd_saved.restype = ctypes.c_int
            lib.gdn_fwd_noalloc.argtypes = [pp] + [P] * 11 + [P]
            lib.gdn_fwd_noalloc.restype = ctypes.c_int
            lib.gdn_fwd_noalloc_error.argtypes = [P]
            lib.gdn_fwd_noalloc_error.restype = ctypes.c_int
            lib.gdn_workspace_error.argtypes = [P, P]
            lib.gdn_workspace_error.restype = ctypes.c_int
            lib.gdn_status_str.argtypes = [ctypes.c_int]
            lib.gdn_status_str.restype = ctypes.c_char_p
            lib.gdn_version.restype = ctypes.c_char_p
            lib.gdn_debug_set_wait.argtypes = [ctypes.c_int64, ctypes.c_int32]
            lib.gdn_debug_set_wait.restype = None
            lib.gdn_cp_trigger.argtypes = [ctypes.c_int64] * 3
            lib.gdn_cp_trigger.restype = ctypes.c_int
            IP = ctypes.POINTER(ctypes.c_int)
            lib.gdn_cp_plan.argtypes = [pp, IP, IP]
            lib.gdn_cp_plan.restype = ctypes.c_int
            _lib = lib
        return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _io_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported io dtype {dt} (bfloat16 or float32)")


def _cuda(t: Optional[torch.Tensor], name: str, dtype=None) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if dtype is not None and t.dtype != dtype:
        t = t.to(dtype)
    return t.contiguous()


def _problem(q, v, scale, cu_seqlens, cu_host, cp_mode, warmup_chunks, out_f32=False):
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    pr = _Problem()
    pr.B, pr.T, pr.Hq, pr.Hv, pr.K, pr.V = B, T, Hq, Hv, K, V
    if cu_seqlens is not None:
        pr.n_seqs = cu_seqlens.numel() - 1
        pr.cu_seqlens = cu_seqlens.data_ptr()
        pr.cu_seqlens_host = cu_host.data_ptr()
    else:
        pr.n_seqs = B
    pr.io_dtype = _io_code(q.dtype)
    pr.scale = float(K ** -0.5 if scale is None else scale)
    pr.cp_mode = CP_MODES[cp_mode] if isinstance(cp_mode, str) else int(cp_mode)
    pr.warmup_chunks = int(warmup_chunks)
    pr.out_f32 = 1 if out_f32 else 0
    return pr


def _cu(cu_seqlens, cu_seqlens_cpu=None):
    if cu_seqlens is None:
        return None, None
    cu = _cuda(cu_seqlens, "cu_seqlens", torch.int32)
    host = cu_seqlens_cpu if cu_seqlens_cpu is not None else cu.cpu()
    host = host.to(torch.int32).contiguous()
    return cu, host


def workspace_bytes(kind: str, q, v, cu_seqlens=None, cu_seqlens_cpu=None, cp_mode="auto",
                    warmup_chunks=8) -> int:
    lib = load_library()
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(q, v, None, cu, host, cp_mode, warmup_chunks)
    fn = {"fwd": lib.gdn_fwd_workspace_bytes, "bwd": lib.gdn_bwd_workspace_bytes,
          "bwd_saved": lib.gdn_bwd_saved_workspace_bytes}[kind]
    return int(fn(ctypes.byref(pr)))


def cp_trigger(n_seqs: int, n_heads: int, seq_len: int) -> bool:
    """Whether the FlashQLA pages' rule turns sequence splitting on."""
    return bool(load_library().gdn_cp_trigger(n_seqs, n_heads, seq_len))


def cp_plan(q, v, cu_seqlens=None, cu_seqlens_cpu=None, cp_mode="warmup", warmup_chunks=8):
    """(seg_len, n_seg) in chunks if the forward would split this problem, else None."""
    lib = load_library()
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(q, v, None, cu, host, cp_mode, warmup_chunks)
    L, n = ctypes.c_int(), ctypes.c_int()
    r = lib.gdn_cp_plan(ctypes.byref(pr), ctypes.byref(L), ctypes.byref(n))
    if r < 0:
        raise ValueError("gdn_cp_plan: bad problem")
    return (L.value, n.value) if r else None


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                               output_final_state=True, output_h=False, output_A=True,
                               cp_mode="auto", warmup_chunks=8, cu_seqlens_cpu=None,
                               workspace: Optional[torch.Tensor] = None, out_f32=False):
    """Returns (g_cum, A, o, h, final_state); h / A / final_state may be None.  ``out_f32`` (bf16
    inputs): o and A come back as fp32, the kernels' values before their final rounding (a checking
    mode; see gdn.h)."""
    lib = load_library()
    io = q.dtype
    q, k, v = _cuda(q, "q", io), _cuda(k, "k", io), _cuda(v, "v", io)
    g, beta = _cuda(g, "g", torch.float32), _cuda(beta, "beta", torch.float32)
    h0 = _cuda(initial_state, "initial_state", torch.float32)
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(q, v, scale, cu, host, cp_mode, warmup_chunks, out_f32)
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    dev = q.device
    odt = torch.float32 if out_f32 else io
    nseq = int(pr.n_seqs)
    nchunks = (sum((int(host[i + 1]) - int(host[i]) + CHUNK - 1) // CHUNK for i in range(nseq))
               if cu is not None else B * ((T + CHUNK - 1) // CHUNK))
    o = torch.empty(B, T, Hv, V, dtype=odt, device=dev)
    g_cum = torch.empty(B, T, Hv, dtype=torch.float32, device=dev)
    A = torch.empty(B, T, Hv, CHUNK, dtype=odt, device=dev) if output_A else None
    h = (torch.empty(nchunks, Hv, K, V, dtype=torch.float32, device=dev) if output_h else None)
    ht = torch.empty(nseq, Hv, K, V, dtype=torch.float32, device=dev) if output_final_state else None
    need = int(lib.gdn_fwd_workspace_bytes(ctypes.byref(pr)))
    if need == 0:
        raise GdnError(1, "gdn_fwd_workspace_bytes")
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    rc = lib.gdn_fwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                     _ptr(g_cum), _ptr(A), _ptr(h), _ptr(ht), _ptr(ws), ws.numel(), ctypes.c_void_p(st))
    if rc != 0:
        raise GdnError(rc, "gdn_fwd")
    if h is not None and cu is None:
        h = h.view(B, (T + CHUNK - 1) // CHUNK, Hv, K, V)
    return g_cum, A, o, h, ht


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, A, do, dht=None, scale=None, initial_state=None,
                               cu_seqlens=None, cu_seqlens_cpu=None,
                               workspace: Optional[torch.Tensor] = None, cp_mode="auto", out_f32=False):
    """``g`` is the forward's returned chunk-local cumsum.  Returns
    (dq, dk, dv, db, dg, dh0); dg is the gradient of the raw gate.  ``cp_mode``
    "auto" splits long sequences of small batch x heads exactly; any other mode
    runs the backward unsplit.  ``out_f32`` (bf16 inputs): dq, dk, dv come back as fp32 (checking
    mode)."""
    lib = load_library()
    io = q.dtype
    q, k, v = _cuda(q, "q", io), _cuda(k, "k", io), _cuda(v, "v", io)
    do = _cuda(do, "do", io)
    g, beta = _cuda(g, "g", torch.float32), _cuda(beta, "beta", torch.float32)
    A = _cuda(A, "A", io)
    h0 = _cuda(initial_state, "initial_state", torch.float32)
    dht = _cuda(dht, "dht", torch.float32)
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(q, v, scale, cu, host, cp_mode, 8, out_f32)
    odt = torch.float32 if out_f32 else io
    dq, dk, dv = (torch.empty(q.shape, dtype=odt, device=q.device), torch.empty(k.shape, dtype=odt, device=q.device),
                  torch.empty(v.shape, dtype=odt, device=q.device))
    db = torch.empty_like(beta)
    dg = torch.empty_like(g)
    dh0 = torch.empty_like(h0) if h0 is not None else None
    need = int(lib.gdn_bwd_workspace_bytes(ctypes.byref(pr)))
    if need == 0:
        raise GdnError(1, "gdn_bwd_workspace_bytes")
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, q.device)
    st = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.gdn_bwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A), _ptr(do),
                     _ptr(dht), _ptr(h0), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(db), _ptr(dg), _ptr(dh0),
                     _ptr(ws), ws.numel(), ctypes.c_void_p(st))
    if rc != 0:
        raise GdnError(rc, "gdn_bwd")
    return dq, dk, dv, db, dg, dh0


class SavedForward:
    """What a forward leaves for its backward: the workspace (operand images and gate vectors of every
    chunk) and the chunk-entry states h (None where the saved backward recomputes, see
    gdn_bwd_saved_uses_saved).  Valid while the forward's inputs are unchanged."""

    def __init__(self, workspace: torch.Tensor, h: Optional[torch.Tensor]):
        self.workspace = workspace
        self.h = h


def chunk_gated_delta_rule_fwd_saved(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                                     output_final_state=True, cp_mode="auto", cu_seqlens_cpu=None,
                                     workspace: Optional[torch.Tensor] = None, out_f32=False):
    """Forward that keeps what its backward needs.  Returns (g_cum, A, o, final_state, saved); pass
    ``saved`` to chunk_gated_delta_rule_bwd_saved, which then skips the backward's recompute passes.
    A given ``workspace`` (large enough) is used and must stay untouched until that backward."""
    lib = load_library()
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(_cuda(q, "q", q.dtype), v, scale, cu, host, cp_mode, 8, out_f32)
    need = int(lib.gdn_fwd_workspace_bytes(ctypes.byref(pr)))
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, q.device)
    # the chunk-entry states are kept only where the saved backward reads them
    keep = int(lib.gdn_bwd_saved_uses_saved(ctypes.byref(pr))) == 1
    g_cum, A, o, h, ht = chunk_gated_delta_rule_fwd(
        q, k, v, g, beta, scale=scale, initial_state=initial_state, cu_seqlens=cu_seqlens,
        output_final_state=output_final_state, output_h=keep, cp_mode=cp_mode, cu_seqlens_cpu=host,
        workspace=ws, out_f32=out_f32)
    return g_cum, A, o, ht, SavedForward(ws, h)


def chunk_gated_delta_rule_bwd_saved(q, k, v, g, beta, A, do, saved: SavedForward, dht=None, scale=None,
                                     initial_state=None, cu_seqlens=None, cu_seqlens_cpu=None, cp_mode="auto",
                                     workspace: Optional[torch.Tensor] = None, out_f32=False):
    """Backward from a chunk_gated_delta_rule_fwd_saved forward on the same inputs (g = its g_cum).
    Returns (dq, dk, dv, db, dg, dh0), equal to chunk_gated_delta_rule_bwd's up to rounding."""
    lib = load_library()
    io = q.dtype
    q, k, v = _cuda(q, "q", io), _cuda(k, "k", io), _cuda(v, "v", io)
    do = _cuda(do, "do", io)
    g, beta = _cuda(g, "g", torch.float32), _cuda(beta, "beta", torch.float32)
    A = _cuda(A, "A", io)
    h0 = _cuda(initial_state, "initial_state", torch.float32)
    dht = _cuda(dht, "dht", torch.float32)
    cu, host = _cu(cu_seqlens, cu_seqlens_cpu)
    pr = _problem(q, v, scale, cu, host, cp_mode, 8, out_f32)
    odt = torch.float32 if out_f32 else io
    dq, dk, dv = (torch.empty(q.shape, dtype=odt, device=q.device), torch.empty(k.shape, dtype=odt, device=q.device),
                  torch.empty(v.shape, dtype=odt, device=q.device))
    db = torch.empty_like(beta)
    dg = torch.empty_like(g)
    dh0 = torch.empty_like(h0) if h0 is not None else None
    need = int(lib.gdn_bwd_saved_workspace_bytes(ctypes.byref(pr)))
    if need == 0:
        raise GdnError(1, "gdn_bwd_saved_workspace_bytes")
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, q.device)
    st = torch.cuda.current_stream(q.device).cuda_stream
    fws = saved.workspace
    rc = lib.gdn_bwd_saved(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A), _ptr(do),
                           _ptr(dht), _ptr(h0), _ptr(saved.h), _ptr(fws), fws.numel(), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(db), _ptr(dg), _ptr(dh0), _ptr(ws), ws.numel(), ctypes.c_void_p(st))
    if rc != 0:
        raise GdnError(rc, "gdn_bwd_saved")
    return dq, dk, dv, db, dg, dh0


class _GdnFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens):
        # keeps the forward's operand images and chunk-entry states for the backward
        g_cum, A, o, ht, saved = chunk_gated_delta_rule_fwd_saved(
            q, k, v, g, beta, scale=scale, initial_state=initial_state, cu_seqlens=cu_seqlens,
            output_final_state=output_final_state)
        ctx.save_for_backward(q, k, v, g_cum, beta, initial_state, cu_seqlens)
        ctx.saved_fwd = saved
        ctx.scale = scale
        ctx.g_dtype, ctx.beta_dtype = g.dtype, beta.dtype
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g_cum, beta, h0, cu = ctx.saved_tensors
        dq, dk, dv, db, dg, dh0 = chunk_gated_delta_rule_bwd_saved(
            q, k, v, g_cum, beta, None, do.contiguous(), ctx.saved_fwd, dht=dht, scale=ctx.scale, initial_state=h0,
            cu_seqlens=cu)
        ctx.saved_fwd = None
        return (dq, dk, dv, dg.to(ctx.g_dtype), db.to(ctx.beta_dtype), None, dh0, None, None)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None,
                           output_final_state=False, cu_seqlens=None):
    """Returns (o, final_state); final_state is None unless requested."""
    o, ht = _GdnFunction.apply(q, k, v, g, beta, scale, initial_state, bool(output_final_state),
                               cu_seqlens)
    return o, (ht if output_final_state else None)
