"""Thin Python binding of libspec_verify.so (ctypes).

Argument marshalling only: every step of verification runs in the library's
CUDA kernels.  Functions take CUDA tensors (contiguous, on one device),
allocate outputs when none are given, and enqueue on the current torch
stream of that device (or ``stream=``, a raw cudaStream_t integer).  There
is no CPU fallback: if the library is missing these functions raise.

The names and argument order follow include/spec_verify.h.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from .build import LIB_PATH

SV_F32, SV_BF16, SV_F16 = 0, 1, 2
_DT = {torch.float32: SV_F32, torch.bfloat16: SV_BF16, torch.float16: SV_F16}

SV_ROW_OK = 0
SV_ROW_BAD_TOKEN = 1
SV_ROW_NONFINITE = 2
SV_ROW_BAD_TREE = 4
SV_ROW_TIMEOUT = 8
SV_ROW_BAD_TEMPERATURE = 16

_lib = None
_lib_lock = threading.Lock()

_VP, _I32P, _F32P = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_INT, _SIZE = ctypes.c_int, ctypes.c_size_t


class SpecVerifyError(RuntimeError):
    """A library call returned a status other than SV_OK."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {spec_verify_status_string(status)}")


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libspec_verify.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libspec_verify.so not found at {LIB_PATH}; build it with "
                    "`python -m speculative_decoding_verification_48_gb300.build` "
                    "(there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            L.spec_verify_workspace_bytes.argtypes = [_INT, _INT, _INT, _INT]
            L.spec_verify_workspace_bytes.restype = _SIZE
            L.spec_verify_chain.argtypes = [_VP, _INT, _VP, _INT, _INT, _I32P, _F32P, _F32P,
                                            _INT, _INT, _INT, _I32P, _I32P, _F32P, _I32P,
                                            _VP, _SIZE, _VP]
            L.spec_verify_chain.restype = _INT
            L.spec_verify_chain_greedy.argtypes = [_VP, _INT, _I32P, _INT, _INT, _INT, _I32P,
                                                   _I32P, _I32P, _VP, _SIZE, _VP]
            L.spec_verify_chain_greedy.restype = _INT
            L.spec_verify_tree_greedy.argtypes = [_VP, _INT, _I32P, _I32P, _INT, _INT, _INT,
                                                  _INT, _I32P, _I32P, _I32P, _I32P, _VP,
                                                  _SIZE, _VP]
            L.spec_verify_tree_greedy.restype = _INT
            L.spec_draft_sample.argtypes = [_VP, _INT, _F32P, _F32P, _INT, _INT, _I32P, _F32P,
                                             _I32P, _VP, _SIZE, _VP]
            L.spec_draft_sample.restype = _INT
            L.spec_tree_mask.argtypes = [_I32P, _INT, _INT, _VP, _I32P, _I32P, _VP]
            L.spec_tree_mask.restype = _INT
            L.spec_tree_kv_compact.argtypes = [_VP, _SIZE, _INT, _INT, _I32P, _I32P, _INT,
                                               _I32P, _I32P, _I32P, _VP]
            L.spec_tree_kv_compact.restype = _INT
            L.spec_verify_wait_selftest.argtypes = [_INT, _VP, _I32P, _VP]
            L.spec_verify_wait_selftest.restype = _INT
            L.spec_verify_force_stream_path.argtypes = [_INT]
            L.spec_verify_force_stream_path.restype = _INT
            L.spec_verify_set_call_counter.argtypes = [ctypes.c_ulonglong]
            L.spec_verify_set_call_counter.restype = ctypes.c_ulonglong
            L.spec_verify_status_string.argtypes = [_INT]
            L.spec_verify_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def spec_verify_status_string(status: int) -> str:
    return lib().spec_verify_status_string(int(status)).decode()


def spec_verify_force_stream_path(on: bool) -> bool:
    """Diagnostics: make every call take the two-launch streaming path
    (on=True) or let small calls take the cluster path (on=False); returns
    the previous setting (see spec_verify_force_stream_path in spec_verify.h)."""
    return bool(lib().spec_verify_force_stream_path(int(bool(on))))


def spec_verify_set_call_counter(calls: int) -> int:
    """Diagnostics: set the library's process-wide call counter; returns the
    previous value (see spec_verify_set_call_counter in spec_verify.h)."""
    return int(lib().spec_verify_set_call_counter(int(calls)))


def spec_verify_workspace_bytes(B: int, rows_per_batch: int, V: int, dtype: int = SV_BF16) -> int:
    return int(lib().spec_verify_workspace_bytes(int(B), int(rows_per_batch), int(V), int(dtype)))


# ---------------------------------------------------------------------------
# Workspace cache: one buffer per (device, stream), grown on demand.  The
# library keeps the 4 KB state header of a workspace valid from call to call,
# so calls of any shape in stream order can share the buffer; a new buffer's
# header is zeroed once, before the first call that uses it.
# ---------------------------------------------------------------------------

_ws_cache: dict = {}
_ws_lock = threading.Lock()


def workspace_for(device: torch.device, stream_ptr: int, nbytes: int) -> torch.Tensor:
    key = (device.index, stream_ptr)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 4096), dtype=torch.uint8, device=device)
            ws[:4096].zero_()
            # the zero-fill ran on torch's current stream; the library call
            # runs on `stream_ptr`, so finish the fill before handing it out
            torch.cuda.current_stream(device).synchronize()
            _ws_cache[key] = ws
        return ws


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def _stream_ptr(device: torch.device, stream) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def spec_verify_chain(target_logits: torch.Tensor, draft: torch.Tensor,
                      draft_tokens: torch.Tensor, temperatures: torch.Tensor,
                      uniforms: torch.Tensor, draft_is_probs: bool = False,
                      out_tokens=None, out_num_accepted=None, out_diag=None,
                      out_row_status=None, want_diag: bool = True, workspace=None,
                      stream=None):
    """Chain speculative sampling (see spec_verify_chain in spec_verify.h).

    Returns (tokens int32 [B, gamma+1], num_accepted int32 [B],
    diag fp32 [B, gamma, 4] or None, row_status int32 [B])."""
    dev = target_logits.device
    B, G1, V = target_logits.shape
    g = G1 - 1
    _check(target_logits, "target_logits", device=dev)
    if target_logits.dtype not in _DT:
        raise TypeError("target_logits dtype must be float32, bfloat16 or float16")
    _check(draft, "draft", shape=(B, g, V), device=dev)
    if draft_is_probs and draft.dtype != torch.float32:
        raise TypeError("draft probabilities must be float32")
    if draft.dtype not in _DT:
        raise TypeError("draft dtype must be float32, bfloat16 or float16")
    _check(draft_tokens, "draft_tokens", torch.int32, (B, g), dev)
    _check(temperatures, "temperatures", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G1), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_diag is None and want_diag:
        out_diag = torch.empty((B, g, 4), dtype=torch.float32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    rows = G1 + (0 if draft_is_probs else g)
    sp = _stream_ptr(dev, stream)
    nbytes = spec_verify_workspace_bytes(B, rows, V, _DT[target_logits.dtype])
    if workspace is None:
        workspace = workspace_for(dev, sp, nbytes)
    st = lib().spec_verify_chain(
        target_logits.data_ptr(), _DT[target_logits.dtype], draft.data_ptr(), _DT[draft.dtype],
        int(bool(draft_is_probs)), draft_tokens.data_ptr(), temperatures.data_ptr(),
        uniforms.data_ptr(), B, g, V, out_tokens.data_ptr(), out_num_accepted.data_ptr(),
        _ptr(out_diag), _ptr(out_row_status), workspace.data_ptr(), workspace.numel(), sp)
    if st != 0:
        raise SpecVerifyError(st, "spec_verify_chain")
    return out_tokens, out_num_accepted, out_diag, out_row_status


def spec_verify_chain_greedy(target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                             out_tokens=None, out_num_accepted=None, out_row_status=None,
                             workspace=None, stream=None):
    """Greedy chain verification.  Returns (tokens, num_accepted, row_status)."""
    dev = target_logits.device
    B, G1, V = target_logits.shape
    g = G1 - 1
    _check(target_logits, "target_logits", device=dev)
    if target_logits.dtype not in _DT:
        raise TypeError("target_logits dtype must be float32, bfloat16 or float16")
    _check(draft_tokens, "draft_tokens", torch.int32, (B, g), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    sp = _stream_ptr(dev, stream)
    nbytes = spec_verify_workspace_bytes(B, G1, V, _DT[target_logits.dtype])
    if workspace is None:
        workspace = workspace_for(dev, sp, nbytes)
    st = lib().spec_verify_chain_greedy(
        target_logits.data_ptr(), _DT[target_logits.dtype], draft_tokens.data_ptr(), B, g, V,
        out_tokens.data_ptr(), out_num_accepted.data_ptr(), _ptr(out_row_status),
        workspace.data_ptr(), workspace.numel(), sp)
    if st != 0:
        raise SpecVerifyError(st, "spec_verify_chain_greedy")
    return out_tokens, out_num_accepted, out_row_status


def spec_verify_tree_greedy(node_logits: torch.Tensor, parent: torch.Tensor,
                            node_tokens: torch.Tensor, max_depth: int, out_path=None,
                            out_tokens=None, out_num_accepted=None, out_row_status=None,
                            workspace=None, stream=None):
    """Token-tree greedy verification.  node_logits is [B, N, V] (or [B*N, V]
    with ``parent`` giving B and N).  Returns (path, tokens, num_accepted,
    row_status)."""
    dev = node_logits.device
    B, N = parent.shape
    V = node_logits.shape[-1]
    _check(node_logits, "node_logits", device=dev)
    if node_logits.numel() != B * N * V:
        raise ValueError("node_logits must hold B*N rows of V entries")
    if node_logits.dtype not in _DT:
        raise TypeError("node_logits dtype must be float32, bfloat16 or float16")
    _check(parent, "parent", torch.int32, (B, N), dev)
    _check(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    W = int(max_depth) + 1
    if out_path is None:
        out_path = torch.empty((B, W), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, W), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    sp = _stream_ptr(dev, stream)
    nbytes = spec_verify_workspace_bytes(B, N, V, _DT[node_logits.dtype])
    if workspace is None:
        workspace = workspace_for(dev, sp, nbytes)
    st = lib().spec_verify_tree_greedy(
        node_logits.data_ptr(), _DT[node_logits.dtype], parent.data_ptr(),
        node_tokens.data_ptr(), B, N, V, int(max_depth), out_path.data_ptr(),
        out_tokens.data_ptr(), out_num_accepted.data_ptr(), _ptr(out_row_status),
        workspace.data_ptr(), workspace.numel(), sp)
    if st != 0:
        raise SpecVerifyError(st, "spec_verify_tree_greedy")
    return out_path, out_tokens, out_num_accepted, out_row_status


def spec_draft_sample(logits: torch.Tensor, temperatures: torch.Tensor, uniforms: torch.Tensor,
                      out_tokens=None, out_probs=None, out_row_status=None, workspace=None,
                      stream=None):
    """Draft-side categorical draw per row (see spec_draft_sample in spec_verify.h).

    logits [B, V] (fp32 / bf16 / fp16, rows 16-byte aligned), temperatures
    fp32 [B], uniforms fp32 [B].  Returns (tokens int32 [B], probs fp32 [B],
    row_status int32 [B])."""
    dev = logits.device
    B, V = logits.shape
    _check(logits, "logits", device=dev)
    if logits.dtype not in _DT:
        raise TypeError("logits dtype must be float32, bfloat16 or float16")
    _check(temperatures, "temperatures", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_probs is None:
        out_probs = torch.empty((B,), dtype=torch.float32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    sp = _stream_ptr(dev, stream)
    nbytes = spec_verify_workspace_bytes(B, 1, V, _DT[logits.dtype])
    if workspace is None:
        workspace = workspace_for(dev, sp, nbytes)
    st = lib().spec_draft_sample(logits.data_ptr(), _DT[logits.dtype], temperatures.data_ptr(),
                                 uniforms.data_ptr(), B, V, out_tokens.data_ptr(),
                                 out_probs.data_ptr(), out_row_status.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), sp)
    if st != 0:
        raise SpecVerifyError(st, "spec_draft_sample")
    return out_tokens, out_probs, out_row_status


def spec_tree_mask(parent: torch.Tensor, out_mask=None, out_depth=None, out_row_status=None,
                   stream=None):
    """Ancestor mask of token trees (see spec_tree_mask in spec_verify.h).

    parent int32 [B, N].  Returns (mask [B, N, ceil(N/64)] as int64 words
    holding the uint64 bit rows, depth int32 [B, N], row_status int32 [B])."""
    dev = parent.device
    B, N = parent.shape
    _check(parent, "parent", torch.int32, (B, N), dev)
    W = (N + 63) // 64
    if out_mask is None:
        out_mask = torch.empty((B, N, W), dtype=torch.int64, device=dev)
    if out_depth is None:
        out_depth = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    st = lib().spec_tree_mask(parent.data_ptr(), B, N, out_mask.data_ptr(), out_depth.data_ptr(),
                              out_row_status.data_ptr(), _stream_ptr(dev, stream))
    if st != 0:
        raise SpecVerifyError(st, "spec_tree_mask")
    return out_mask, out_depth, out_row_status


def spec_tree_kv_compact(kv: torch.Tensor, base: torch.Tensor, path: torch.Tensor,
                         num_accepted: torch.Tensor, out_length=None, out_row_status=None,
                         stream=None):
    """Move each tree's accepted-path KV rows to contiguous slots, in place
    (see spec_tree_kv_compact in spec_verify.h).

    kv [B, S, ...] contiguous, any dtype, each [S] row a multiple of 16 bytes;
    base, num_accepted int32 [B]; path int32 [B, Wp].  Returns (length [B],
    row_status [B])."""
    dev = kv.device
    B, S = kv.shape[:2]
    _check(kv, "kv", device=dev)
    row_bytes = (kv.numel() // (B * S)) * kv.element_size() if B * S else 0
    _check(base, "base", torch.int32, (B,), dev)
    _check(num_accepted, "num_accepted", torch.int32, (B,), dev)
    if path.dim() != 2 or path.shape[0] != B:
        raise ValueError("path must be [B, Wp]")
    _check(path, "path", torch.int32, tuple(path.shape), dev)
    if out_length is None:
        out_length = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_row_status is None:
        out_row_status = torch.empty((B,), dtype=torch.int32, device=dev)
    st = lib().spec_tree_kv_compact(kv.data_ptr(), row_bytes, B, S, base.data_ptr(),
                                    path.data_ptr(), path.shape[1], num_accepted.data_ptr(),
                                    out_length.data_ptr(), out_row_status.data_ptr(),
                                    _stream_ptr(dev, stream))
    if st != 0:
        raise SpecVerifyError(st, "spec_tree_kv_compact")
    return out_length, out_row_status


def spec_verify_wait_selftest(which: int, device=None, stream=None) -> int:
    """Run bounded wait ``which`` (0: counter reset, 1: the decide kernel's
    poll of tagged partials) on words that nothing sets (see
    spec_verify_wait_selftest in spec_verify.h);
    returns the status the device reported, SV_ROW_TIMEOUT when the wait gave
    up as it should."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    scratch = torch.empty(64, dtype=torch.uint8, device=dev)
    out = torch.full((1,), -1, dtype=torch.int32, device=dev)
    sp = _stream_ptr(dev, stream)
    st = lib().spec_verify_wait_selftest(int(which), scratch.data_ptr(), out.data_ptr(), sp)
    if st != 0:
        raise SpecVerifyError(st, "spec_verify_wait_selftest")
    torch.cuda.synchronize(dev)
    return int(out.item())
