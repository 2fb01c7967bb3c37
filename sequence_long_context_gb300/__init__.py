"""GB300-native sequence-parallel attention core (Python binding).

The functions named usp_* mirror the C ABI of include/usp.h one to one and
only marshal arguments (tensors -> device pointers, the current CUDA stream).
Every step of the computation runs in the CUDA library libusp.so; there is
no Python or CPU fallback, and a missing library raises.

The helpers below them (attn_forward, attn_backward, permute,
merge_partials) allocate outputs and workspaces with PyTorch and call the
same entry points.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import _lib

LAYOUT = {"contiguous": 0, "zigzag": 1, "stripe": 2}
DTYPE = {torch.bfloat16: 0, torch.float32: 1}
PERMUTE = {"extract": 0, "restore": 1, "seq2head": 2, "head2seq": 3}
FLAG_FORCE_SIMT = 1
FLAG_SAVED_EXCHANGE = 2
FLAG_NATURAL_ORDER = 4


class UspError(RuntimeError):
    pass


def _p(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr() if x.numel() else None
    return int(x)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _check(status: int) -> None:
    if status != 0:
        lib = _lib.load()
        name = lib.usp_status_string(status).decode()
        if name == "USP_ERR_CUDA":
            name += ": " + lib.usp_last_error_detail().decode()
        raise UspError(name)


def _enum(table, x) -> int:
    return table[x] if not isinstance(x, int) else x


# --- the C ABI, one to one ---------------------------------------------------

def usp_attn_fwd(q, k, v, out, lse, B, S, Hq, Hkv, D, softmax_scale, causal,
                 window, sink_tokens, cu_seqlens, cp_size, ulysses_degree,
                 layout, dtype, flags=0, workspace=None, workspace_bytes=0,
                 stream=None) -> None:
    _check(_lib.load().usp_attn_fwd(
        _p(q), _p(k), _p(v), _p(out), _p(lse), B, S, Hq, Hkv, D,
        float(softmax_scale), int(causal), int(window), int(sink_tokens),
        _p(cu_seqlens), cp_size, ulysses_degree, _enum(LAYOUT, layout),
        _enum(DTYPE, dtype), flags, _p(workspace), int(workspace_bytes),
        _stream(stream)))


def usp_attn_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, out, lse, B, S, Hq, Hkv,
                     D, softmax_scale, causal, window, sink_tokens, cu_seqlens, cp_size,
                     ulysses_degree, layout, flags=0, workspace=None, workspace_bytes=0,
                     stream=None) -> None:
    _check(_lib.load().usp_attn_fwd_fp8(
        _p(q), _p(k), _p(v), float(q_descale), float(k_descale), float(v_descale), _p(out),
        _p(lse), B, S, Hq, Hkv, D, float(softmax_scale), int(causal), int(window),
        int(sink_tokens), _p(cu_seqlens), cp_size, ulysses_degree, _enum(LAYOUT, layout),
        flags, _p(workspace), int(workspace_bytes), _stream(stream)))


def usp_attn_fwd_fp8_workspace_size(B, S, Hq, Hkv, D, cp_size, ulysses_degree) -> int:
    return int(_lib.load().usp_attn_fwd_fp8_workspace_size(B, S, Hq, Hkv, D, cp_size,
                                                           ulysses_degree))


def usp_quantize_e4m3(x, out, n, inv_scale, stream=None) -> None:
    _check(_lib.load().usp_quantize_e4m3(_p(x), _p(out), int(n), float(inv_scale),
                                         _stream(stream)))


def usp_attn_fwd_workspace_size(B, S, Hq, Hkv, D, cp_size, ulysses_degree,
                                dtype, flags=0) -> int:
    return int(_lib.load().usp_attn_fwd_workspace_size(
        B, S, Hq, Hkv, D, cp_size, ulysses_degree, _enum(DTYPE, dtype), flags))


def usp_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D,
                 softmax_scale, causal, window, sink_tokens, cu_seqlens,
                 cp_size, ulysses_degree, layout, dtype, flags=0,
                 workspace=None, workspace_bytes=0, stream=None) -> None:
    _check(_lib.load().usp_attn_bwd(
        _p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk),
        _p(dv), B, S, Hq, Hkv, D, float(softmax_scale), int(causal),
        int(window), int(sink_tokens), _p(cu_seqlens), cp_size,
        ulysses_degree, _enum(LAYOUT, layout), _enum(DTYPE, dtype), flags,
        _p(workspace), int(workspace_bytes), _stream(stream)))


def usp_attn_bwd_workspace_size(B, S, Hq, Hkv, D, cp_size, ulysses_degree,
                                dtype, flags=0) -> int:
    return int(_lib.load().usp_attn_bwd_workspace_size(
        B, S, Hq, Hkv, D, cp_size, ulysses_degree, _enum(DTYPE, dtype), flags))


def usp_attn_bwd_noalloc(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv,
                         D, softmax_scale, causal, window, sink_tokens,
                         cu_seqlens, cp_size, ulysses_degree, layout, dtype,
                         flags=0, stream=None) -> None:
    """usp_attn_bwd without a workspace: scratch comes from the library's
    fixed 64 MiB device array (for callers that cannot allocate; calls that
    overlap on the GPU race on it)."""
    _check(_lib.load().usp_attn_bwd_noalloc(
        _p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk),
        _p(dv), B, S, Hq, Hkv, D, float(softmax_scale), int(causal),
        int(window), int(sink_tokens), _p(cu_seqlens), cp_size,
        ulysses_degree, _enum(LAYOUT, layout), _enum(DTYPE, dtype), flags,
        _stream(stream)))


def usp_merge_partials(o_parts, lse_parts, n, rows, D, tree_order, o_out,
                       out_dtype, lse_out, stream=None) -> None:
    _check(_lib.load().usp_merge_partials(
        _p(o_parts), _p(lse_parts), n, rows, D, int(tree_order), _p(o_out),
        _enum(DTYPE, out_dtype), _p(lse_out), _stream(stream)))


def usp_attn_decode(q, k, v, out, lse, B, Tq, S, Hq, Hkv, D, softmax_scale,
                    causal, cp_size, splits_per_shard, tree_order, dtype,
                    workspace=None, workspace_bytes=0, stream=None) -> None:
    _check(_lib.load().usp_attn_decode(
        _p(q), _p(k), _p(v), _p(out), _p(lse), B, Tq, S, Hq, Hkv, D,
        float(softmax_scale), int(causal), cp_size, splits_per_shard,
        int(tree_order), _enum(DTYPE, dtype), _p(workspace),
        int(workspace_bytes), _stream(stream)))


def usp_attn_decode_workspace_size(B, Tq, S, Hq, Hkv, D, cp_size,
                                   splits_per_shard) -> int:
    return int(_lib.load().usp_attn_decode_workspace_size(
        B, Tq, S, Hq, Hkv, D, cp_size, splits_per_shard))


def usp_permute(src, dst, kind, layout, B, S, H, D, cp_size, ulysses_degree,
                elem_bytes, stream=None) -> None:
    _check(_lib.load().usp_permute(
        _p(src), _p(dst), _enum(PERMUTE, kind), _enum(LAYOUT, layout), B, S, H,
        D, cp_size, ulysses_degree, elem_bytes, _stream(stream)))


def usp_check_cu_seqlens(cu_seqlens_host, nseq, total_tokens) -> None:
    """Raise unless cu_seqlens_host (int32, host) starts at 0, never
    decreases and ends at total_tokens (the debug-mode check)."""
    st = _lib.load().usp_check_cu_seqlens(_p(cu_seqlens_host), int(nseq), int(total_tokens))
    if st != 0:
        lib = _lib.load()
        raise UspError(lib.usp_status_string(st).decode() + ": "
                       + lib.usp_last_error_detail().decode())


def usp_launch_count() -> int:
    return int(_lib.load().usp_launch_count())


def usp_device_status() -> None:
    """Raise if a kernel flagged a failed (timed-out) wait since the last call."""
    _check(_lib.load().usp_device_status())


def usp_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch a kernel whose bounded wait must time out after limit_us
    (diagnostics: the next usp_device_status() reports USP_ERR_TIMEOUT)."""
    _check(_lib.load().usp_selftest_wait_timeout(int(limit_us), _stream(stream)))


def usp_profile_enable(on: bool) -> None:
    _check(_lib.load().usp_profile_enable(int(bool(on))))


def usp_profile_read(max_stats: int = 64) -> dict:
    """{kernel name: (launches, total device ms)} since the last read."""
    arr = (_lib.KernelStat * max_stats)()
    n = _lib.load().usp_profile_read(arr, max_stats)
    if n < 0:
        raise UspError("USP_ERR_CUDA")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(n)}


# --- allocation helpers -----------------------------------------------------

def _dims(q: torch.Tensor, k: torch.Tensor, cu_seqlens):
    if cu_seqlens is not None:
        T, Hq, D = q.shape
        return int(cu_seqlens.numel() - 1), T, Hq, k.shape[1], D, 1
    B, S, Hq, D = q.shape
    return B, S, Hq, k.shape[2], D, B


def _packed_dims(qkv: torch.Tensor, cu_seqlens):
    if cu_seqlens is not None:
        T, _, H, D = qkv.shape
        return int(cu_seqlens.numel() - 1), T, H, D, 1
    B, S, _, H, D = qkv.shape
    return B, S, H, D, B


def check_cu_seqlens(cu_seqlens: torch.Tensor, total_tokens: int) -> None:
    """Check packed-sequence boundaries on the host before a call (the
    attention calls trust them); copies a device tensor to the host."""
    cu = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    if cu.dim() != 1 or cu.numel() < 2:
        raise UspError("USP_ERR_INVALID_ARG: cu_seqlens needs at least two entries")
    usp_check_cu_seqlens(cu, cu.numel() - 1, total_tokens)


def attn_forward_qkvpacked(qkv, *, causal=True, window=0, sink_tokens=0,
                           cu_seqlens=None, cp=1, ud=1, layout="contiguous",
                           softmax_scale=0.0, flags=0, workspace=None, stream=None):
    """(out, lse) for a packed rank-major qkv [B,S,3,H,D] (packed sequences:
    [T,3,H,D] with cu_seqlens)."""
    B, S, H, D, Bl = _packed_dims(qkv, cu_seqlens)
    out = torch.empty(qkv.shape[:-3] + (H, D), dtype=qkv.dtype, device=qkv.device)
    lse = torch.empty((Bl, H, S) if cu_seqlens is None else (H, S),
                      dtype=torch.float32, device=qkv.device)
    ws, ws_n = _use_workspace(
        workspace, usp_attn_fwd_workspace_size(Bl, S, H, H, D, cp, ud, qkv.dtype, flags),
        qkv.device)
    _check(_lib.load().usp_attn_fwd_qkvpacked(
        _p(qkv), _p(out), _p(lse), B, S, H, D, float(softmax_scale), int(causal),
        int(window), int(sink_tokens), _p(cu_seqlens), cp, ud, _enum(LAYOUT, layout),
        _enum(DTYPE, qkv.dtype), flags, _p(ws), int(ws_n), _stream(stream)))
    return out, lse


def attn_backward_qkvpacked(qkv, out, lse, dout, *, causal=True, window=0,
                            sink_tokens=0, cu_seqlens=None, cp=1, ud=1,
                            layout="contiguous", softmax_scale=0.0, flags=0,
                            workspace=None, saved_exchange=False,
                            stream=None) -> torch.Tensor:
    """dqkv (qkv's shape) for a packed qkv and the forward's (out, lse);
    saved_exchange as in attn_backward."""
    B, S, H, D, Bl = _packed_dims(qkv, cu_seqlens)
    dqkv = torch.empty_like(qkv)
    if saved_exchange:
        if workspace is None:
            raise ValueError("saved_exchange needs the forward's workspace")
        flags |= FLAG_SAVED_EXCHANGE
    ws, ws_n = _use_workspace(
        workspace, usp_attn_bwd_workspace_size(Bl, S, H, H, D, cp, ud, qkv.dtype, flags),
        qkv.device)
    _check(_lib.load().usp_attn_bwd_qkvpacked(
        _p(qkv), _p(out), _p(lse), _p(dout), _p(dqkv), B, S, H, D,
        float(softmax_scale), int(causal), int(window), int(sink_tokens),
        _p(cu_seqlens), cp, ud, _enum(LAYOUT, layout), _enum(DTYPE, qkv.dtype),
        flags, _p(ws), int(ws_n), _stream(stream)))
    return dqkv


def attn_decode(q, k, v, *, causal=True, cp=1, splits=1, tree_order=True,
                softmax_scale=0.0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """(out [B,Tq,Hq,D], lse [B,Tq,Hq]) of the newest Tq tokens q
    [B,Tq,Hq,D] against a rank-major contiguous KV cache k, v [B,S,Hkv,D]."""
    B, Tq, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    out = torch.empty_like(q)
    lse = torch.empty((B, Tq, Hq), dtype=torch.float32, device=q.device)
    ws_n = usp_attn_decode_workspace_size(B, Tq, S, Hq, Hkv, D, cp, splits)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=q.device)
    usp_attn_decode(q, k, v, out, lse, B, Tq, S, Hq, Hkv, D, softmax_scale,
                    causal, cp, splits, tree_order, q.dtype, ws, ws_n, stream)
    return out, lse


def _use_workspace(workspace, need, device):
    """The caller's uint8 workspace (checked for size), else a fresh one."""
    if workspace is None:
        return torch.empty(need, dtype=torch.uint8, device=device) if need else None, need
    if workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    return workspace, workspace.numel()


def attn_workspace(q, k, *, cu_seqlens=None, cp=1, ud=1, flags=0,
                   natural=False) -> torch.Tensor:
    """A workspace that fits both attn_forward and attn_backward of these
    shapes. Passing the same one to both, and saved_exchange=True to the
    backward, lets the backward reuse the forward's Ulysses exchange (or,
    natural=True, its rank-major copies)."""
    if natural:
        flags |= FLAG_NATURAL_ORDER
    B, S, Hq, Hkv, D, Bl = _dims(q, k, cu_seqlens)
    n = usp_attn_bwd_workspace_size(Bl, S, Hq, Hkv, D, cp, ud, q.dtype, flags)
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def attn_forward(q, k, v, *, causal=True, window=0, sink_tokens=0,
                 cu_seqlens=None, cp=1, ud=1, layout="contiguous",
                 softmax_scale=0.0, flags=0, workspace=None, stream=None,
                 natural=False) -> Tuple[torch.Tensor, torch.Tensor]:
    """(out, lse) for rank-major q/k/v ([B,S,H,D] or packed [T,H,D]);
    natural=True: q/k/v and out in natural sequence order (lse rank-major),
    the layout's extract and restore done inside the call
    (FLAG_NATURAL_ORDER)."""
    if natural:
        flags |= FLAG_NATURAL_ORDER
    B, S, Hq, Hkv, D, Bl = _dims(q, k, cu_seqlens)
    out = torch.empty_like(q)
    lse = torch.empty((Bl, Hq, S) if cu_seqlens is None else (Hq, S),
                      dtype=torch.float32, device=q.device)
    ws, ws_n = _use_workspace(
        workspace, usp_attn_fwd_workspace_size(Bl, S, Hq, Hkv, D, cp, ud, q.dtype, flags),
        q.device)
    usp_attn_fwd(q, k, v, out, lse, B, S, Hq, Hkv, D, softmax_scale, causal,
                 window, sink_tokens, cu_seqlens, cp, ud, layout, q.dtype,
                 flags, ws, ws_n, stream)
    return out, lse


def attn_backward(q, k, v, out, lse, dout, *, causal=True, window=0,
                  sink_tokens=0, cu_seqlens=None, cp=1, ud=1,
                  layout="contiguous", softmax_scale=0.0, flags=0,
                  workspace=None, saved_exchange=False, stream=None, natural=False):
    """(dq, dk, dv) for rank-major tensors and the forward's (out, lse).
    saved_exchange: workspace is the one the forward wrote (attn_workspace),
    holding its head-sharded q, k, v, out (FLAG_SAVED_EXCHANGE).
    natural: as in attn_forward (every tensor but lse in natural order)."""
    if natural:
        flags |= FLAG_NATURAL_ORDER
    B, S, Hq, Hkv, D, Bl = _dims(q, k, cu_seqlens)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if saved_exchange:
        if workspace is None:
            raise ValueError("saved_exchange needs the forward's workspace")
        flags |= FLAG_SAVED_EXCHANGE
    ws, ws_n = _use_workspace(
        workspace, usp_attn_bwd_workspace_size(Bl, S, Hq, Hkv, D, cp, ud, q.dtype, flags),
        q.device)
    usp_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, S, Hq, Hkv, D,
                 softmax_scale, causal, window, sink_tokens, cu_seqlens, cp,
                 ud, layout, q.dtype, flags, ws, ws_n, stream)
    return dq, dk, dv


def quantize_e4m3(x: torch.Tensor, inv_scale: float, stream=None) -> torch.Tensor:
    """E4M3 codes (uint8, x's shape) of a bf16 tensor times inv_scale."""
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("quantize_e4m3 takes a contiguous bf16 tensor")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    usp_quantize_e4m3(x, out, x.numel(), inv_scale, stream)
    return out


def attn_forward_fp8(q8, k8, v8, q_descale, k_descale, v_descale, *, causal=True,
                     window=0, sink_tokens=0, cu_seqlens=None, cp=1, ud=1,
                     layout="contiguous", softmax_scale=0.0, workspace=None, stream=None
                     ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(out bf16, lse) for rank-major e4m3 codes q8/k8/v8 (uint8 or
    float8_e4m3fn tensors, [B,S,H,128] or packed [T,H,128]) with per-tensor
    descales."""
    B, S, Hq, Hkv, D, Bl = _dims(q8, k8, cu_seqlens)
    out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((Bl, Hq, S) if cu_seqlens is None else (Hq, S),
                      dtype=torch.float32, device=q8.device)
    ws, ws_n = _use_workspace(
        workspace, usp_attn_fwd_fp8_workspace_size(Bl, S, Hq, Hkv, D, cp, ud), q8.device)
    usp_attn_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, out, lse, B, S, Hq, Hkv,
                     D, softmax_scale, causal, window, sink_tokens, cu_seqlens, cp, ud,
                     layout, 0, ws, ws_n, stream)
    return out, lse


def permute(x: torch.Tensor, kind: str, layout: str = "contiguous", cp: int = 1,
            ud: int = 1, stream=None) -> torch.Tensor:
    """Layout extract/restore of [B,S,H,D] (packed: [T,H,D]) or the Ulysses
    exchange ([B,S,H,D] <-> [ud,B,S,H/ud,D])."""
    if kind in ("extract", "restore"):
        xb = x if x.dim() == 4 else x.unsqueeze(0)
        B, S, H, D = xb.shape
        dst = torch.empty_like(x)
    elif kind == "seq2head":
        B, S, H, D = x.shape
        dst = torch.empty((ud, B, S, H // ud, D), dtype=x.dtype, device=x.device)
    else:
        _, B, S, Hg, D = x.shape
        H = Hg * ud
        dst = torch.empty((B, S, H, D), dtype=x.dtype, device=x.device)
    usp_permute(x, dst, kind, layout, B, S, H, D, cp, ud, x.element_size(),
                stream)
    return dst


def merge_partials(o_parts: torch.Tensor, lse_parts: torch.Tensor,
                   tree_order: bool = False, out_dtype=torch.float32,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """o_parts [n, rows, D] fp32, lse_parts [n, rows] -> (O [rows, D], LSE)."""
    n, rows, D = o_parts.shape
    o = torch.empty((rows, D), dtype=out_dtype, device=o_parts.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    usp_merge_partials(o_parts, lse_parts, n, rows, D, tree_order, o,
                       out_dtype, lse, stream)
    return o, lse
