"""Python binding of libspecverify (argument marshalling only).

Every function here has the name of the C entry point it calls and does nothing but check
tensor types, shapes and devices, take raw device pointers and the current CUDA stream from
PyTorch, and forward them.  All of the verification runs in the library's CUDA kernels; if
the shared library is missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

SPEC_BF16 = 0
SPEC_F32 = 1
SPEC_MAX_GAMMA = 32
ST_BAD_DRAFT, ST_R_ZERO, ST_CLAMPED_GAMMA, ST_HISTORY_FULL = 1, 2, 4, 8
ST_TIMEOUT, ST_STOPPED, ST_BAD_TREE, ST_BAD_ROW = 16, 32, 64, 128

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libspecverify.so (built in-tree by build.build()); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise SpecVerifyError(f"{p} is missing: build it with "
                              "speculative_decoding_verification_34_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    size_t = ctypes.c_size_t
    lib.spec_verify_greedy.argtypes = [vp, i32, vp, vp, sz, sz, sz, vp, vp, vp, vp, size_t, vp]
    lib.spec_verify_greedy.restype = i32
    lib.spec_verify_sample.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp, size_t, vp]
    lib.spec_verify_sample.restype = i32
    lib.spec_verify_greedy_split.argtypes = [vp, vp, i32, vp, vp, sz, sz, sz, vp, vp, vp, vp, size_t, vp]
    lib.spec_verify_greedy_split.restype = i32
    lib.spec_verify_sample_split.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp,
                                             size_t, vp]
    lib.spec_verify_sample_split.restype = i32
    lib.spec_verify_tree_greedy.argtypes = [vp, i32, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp, size_t, vp]
    lib.spec_verify_sample_truncated.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp,
                                                 vp, size_t, vp]
    lib.spec_verify_sample_truncated.restype = i32
    lib.spec_verify_sample_truncated_split.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, sz, sz, vp,
                                                       vp, vp, vp, vp, size_t, vp]
    lib.spec_verify_sample_truncated_split.restype = i32
    lib.spec_verify_tree_greedy.restype = i32
    lib.spec_verify_tree_greedy_commit.argtypes = [vp, i32, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp, size_t,
                                                   vp, vp, i32, vp, vp, sz, vp]
    lib.spec_verify_tree_greedy_commit.restype = i32
    lib.spec_verify_sample_static.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp]
    lib.spec_verify_greedy_commit.argtypes = [vp, i32, vp, vp, sz, sz, sz, vp, vp, vp, vp, size_t,
                                              vp, vp, i32, vp, vp, sz, vp]
    lib.spec_verify_greedy_commit.restype = i32
    lib.spec_verify_sample_commit.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp, vp, vp, vp,
                                              size_t, vp, vp, i32, vp, vp, sz, vp]
    lib.spec_verify_sample_commit.restype = i32
    lib.spec_verify_sample_truncated_commit.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, sz, sz, vp, vp,
                                                        vp, vp, vp, size_t, vp, vp, i32, vp, vp, sz, vp]
    lib.spec_verify_sample_truncated_commit.restype = i32
    lib.spec_verify_sample_static.restype = i32
    lib.spec_verify_workspace_bytes.argtypes = [sz, sz, sz, i32]
    lib.spec_verify_workspace_bytes.restype = size_t
    lib.spec_commit_kv_lengths.argtypes = [vp, sz, vp, vp, i32, vp, sz, vp, vp, sz, vp, vp]
    lib.spec_commit_kv_lengths.restype = i32
    lib.spec_apply_stops.argtypes = [vp, vp, sz, sz, i32, vp, vp, vp]
    lib.spec_apply_stops.restype = i32
    lib.spec_last_error.argtypes = []
    lib.spec_last_error.restype = ctypes.c_char_p
    lib.spec_launch_count.argtypes = []
    lib.spec_launch_count.restype = ctypes.c_uint64
    lib.spec_verify_plan.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.spec_verify_plan.restype = i32
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        msg = load_library().spec_last_error().decode(errors="replace")
        raise SpecVerifyError(f"specverify error {rc}: {msg}")


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def spec_verify_workspace_bytes(B: int, gmax: int, V: int, dtype: int = SPEC_BF16) -> int:
    return int(load_library().spec_verify_workspace_bytes(B, gmax, V, dtype))


def alloc_workspace(B: int, gmax: int, V: int, dtype: int = SPEC_BF16, device=None) -> torch.Tensor:
    """A zero-filled device workspace for verify calls of these sizes (reusable: every call
    returns its counters to zero; one call at a time)."""
    n = spec_verify_workspace_bytes(B, gmax, V, dtype)
    return torch.zeros(max(n, 64), dtype=torch.uint8, device=device or "cuda")


def _ws(workspace, B, gmax, V, code, device):
    if workspace is None:
        workspace = alloc_workspace(B, gmax, V, code, device)
    if workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    return workspace, _ptr(workspace, "workspace"), workspace.numel()


def spec_verify_greedy(target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                       num_draft: Optional[torch.Tensor], out_tokens: torch.Tensor,
                       num_accepted: torch.Tensor, status: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    lib = load_library()
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    _check(lib.spec_verify_greedy(
        _ptr(target_logits, "target_logits"), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def spec_verify_sample(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                       draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                       temperature: torch.Tensor, u_accept: torch.Tensor, u_sample: torch.Tensor,
                       out_tokens: torch.Tensor, num_accepted: torch.Tensor,
                       diag: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    lib = load_library()
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    _check(lib.spec_verify_sample(
        _ptr(target_logits, "target_logits"),
        _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)),
        _ptr(temperature, "temperature", torch.float32, (B,)),
        _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
        _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def _commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len):
    cap = history.shape[1] if history is not None else 0
    return (_ptr(target_kv_len, "target_kv_len", torch.int32, (B,)),
            _ptr(draft_kv_len, "draft_kv_len", torch.int32, (B,)), int(bool(correction_processed)),
            _ptr(history, "history", torch.int32), _ptr(committed_len, "committed_len", torch.int32, (B,)), cap)


def spec_verify_greedy_commit(target_logits: torch.Tensor, draft_tokens: torch.Tensor,
                              num_draft: Optional[torch.Tensor], out_tokens: torch.Tensor,
                              num_accepted: torch.Tensor, target_kv_len: torch.Tensor,
                              draft_kv_len: Optional[torch.Tensor] = None, correction_processed: bool = True,
                              history: Optional[torch.Tensor] = None, committed_len: Optional[torch.Tensor] = None,
                              status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                              stream=None) -> None:
    """spec_verify_greedy and spec_commit_kv_lengths of the same round in one launch."""
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    lib = load_library()
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    _check(lib.spec_verify_greedy_commit(
        _ptr(target_logits, "target_logits"), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn,
        *_commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len),
        _stream(stream)))


def _sample_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept, u_sample,
                        out_tokens, num_accepted, diag, status, workspace, target_kv_len, draft_kv_len,
                        correction_processed, history, committed_len, stream):
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    args = (_ptr(target_logits, "target_logits"),
            _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)),
            _ptr(temperature, "temperature", torch.float32, (B,)),
            _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
            _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn,
            *_commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len),
            _stream(stream))
    return args, ws


def spec_verify_sample_commit(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                              draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                              temperature: torch.Tensor, u_accept: torch.Tensor, u_sample: torch.Tensor,
                              out_tokens: torch.Tensor, num_accepted: torch.Tensor, target_kv_len: torch.Tensor,
                              draft_kv_len: Optional[torch.Tensor] = None, correction_processed: bool = True,
                              history: Optional[torch.Tensor] = None, committed_len: Optional[torch.Tensor] = None,
                              diag: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample and spec_commit_kv_lengths of the same round in one launch."""
    args, _ = _sample_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept,
                                  u_sample, out_tokens, num_accepted, diag, status, workspace, target_kv_len,
                                  draft_kv_len, correction_processed, history, committed_len, stream)
    _check(load_library().spec_verify_sample_commit(*args))


def spec_verify_sample_truncated(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                                 draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                                 temperature: torch.Tensor, top_k: Optional[torch.Tensor],
                                 top_p: Optional[torch.Tensor], u_accept: torch.Tensor, u_sample: torch.Tensor,
                                 out_tokens: torch.Tensor, num_accepted: torch.Tensor,
                                 diag: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample on top-k / top-p truncated distributions (top_k int32 [B], top_p
    float32 [B], either None); bf16 logits."""
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    lib = load_library()
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    _check(lib.spec_verify_sample_truncated(
        _ptr(target_logits, "target_logits"),
        _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)),
        _ptr(temperature, "temperature", torch.float32, (B,)),
        _ptr(top_k, "top_k", torch.int32, (B,)), _ptr(top_p, "top_p", torch.float32, (B,)),
        _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
        _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def _truncated_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k, top_p,
                           u_accept, u_sample, out_tokens, num_accepted, diag, status, workspace, target_kv_len,
                           draft_kv_len, correction_processed, history, committed_len, stream):
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    args = (_ptr(target_logits, "target_logits"),
            _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)),
            _ptr(temperature, "temperature", torch.float32, (B,)),
            _ptr(top_k, "top_k", torch.int32, (B,)), _ptr(top_p, "top_p", torch.float32, (B,)),
            _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
            _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn,
            *_commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len),
            _stream(stream))
    return args, ws


def spec_verify_sample_truncated_commit(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                                        draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                                        temperature: torch.Tensor, top_k: Optional[torch.Tensor],
                                        top_p: Optional[torch.Tensor], u_accept: torch.Tensor,
                                        u_sample: torch.Tensor, out_tokens: torch.Tensor,
                                        num_accepted: torch.Tensor, target_kv_len: torch.Tensor,
                                        draft_kv_len: Optional[torch.Tensor] = None,
                                        correction_processed: bool = True, history: Optional[torch.Tensor] = None,
                                        committed_len: Optional[torch.Tensor] = None,
                                        diag: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                        workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample_truncated and spec_commit_kv_lengths of the same round, fused."""
    args, _ = _truncated_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k,
                                     top_p, u_accept, u_sample, out_tokens, num_accepted, diag, status, workspace,
                                     target_kv_len, draft_kv_len, correction_processed, history, committed_len,
                                     stream)
    _check(load_library().spec_verify_sample_truncated_commit(*args))


def spec_verify_sample_truncated_split(saved_logits: torch.Tensor, block_logits: Optional[torch.Tensor],
                                       draft_logits: torch.Tensor, draft_tokens: torch.Tensor,
                                       num_draft: Optional[torch.Tensor], temperature: torch.Tensor,
                                       top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
                                       u_accept: torch.Tensor, u_sample: torch.Tensor, out_tokens: torch.Tensor,
                                       num_accepted: torch.Tensor, diag: Optional[torch.Tensor] = None,
                                       status: Optional[torch.Tensor] = None,
                                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample_truncated with target row 0 (saved_logits [B][V]) apart from rows
    1..gmax (block_logits [B][gmax][V])."""
    B, gmax, V = _split_shapes(saved_logits, block_logits)
    if draft_logits.dtype != saved_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    lib = load_library()
    code = _dtype_code(saved_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, saved_logits.device)
    _check(lib.spec_verify_sample_truncated_split(
        _ptr(saved_logits, "saved_logits"), _ptr(block_logits, "block_logits"),
        _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)),
        _ptr(temperature, "temperature", torch.float32, (B,)),
        _ptr(top_k, "top_k", torch.int32, (B,)), _ptr(top_p, "top_p", torch.float32, (B,)),
        _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
        _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def spec_verify_tree_greedy(target_logits: torch.Tensor, node_tokens: torch.Tensor,
                            node_parents: torch.Tensor, num_nodes: Optional[torch.Tensor],
                            out_tokens: torch.Tensor, num_accepted: torch.Tensor,
                            path_nodes: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Greedy verification of draft trees: target_logits [B][nmax+1][V] (row j after node j),
    node_tokens and node_parents [B][nmax] (node j+1's token and parent, parent < j+1)."""
    B, np1, V = target_logits.shape
    nmax = np1 - 1
    lib = load_library()
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, nmax, V, code, target_logits.device)
    _check(lib.spec_verify_tree_greedy(
        _ptr(target_logits, "target_logits"), code,
        _ptr(node_tokens, "node_tokens", torch.int32, (B, nmax)),
        _ptr(node_parents, "node_parents", torch.int32, (B, nmax)),
        _ptr(num_nodes, "num_nodes", torch.int32, (B,)), B, nmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, nmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(path_nodes, "path_nodes", torch.int32, (B, nmax)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def _tree_args(target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted, path_nodes, status,
               workspace):
    B, np1, V = target_logits.shape
    nmax = np1 - 1
    ws, wsp, wsn = _ws(workspace, B, nmax, V, _dtype_code(target_logits), target_logits.device)
    args = (_ptr(target_logits, "target_logits"), _dtype_code(target_logits),
            _ptr(node_tokens, "node_tokens", torch.int32, (B, nmax)),
            _ptr(node_parents, "node_parents", torch.int32, (B, nmax)),
            _ptr(num_nodes, "num_nodes", torch.int32, (B,)), B, nmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, nmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(path_nodes, "path_nodes", torch.int32, (B, nmax)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn)
    return args, ws


def spec_verify_tree_greedy_commit(target_logits: torch.Tensor, node_tokens: torch.Tensor,
                                   node_parents: torch.Tensor, num_nodes: Optional[torch.Tensor],
                                   out_tokens: torch.Tensor, num_accepted: torch.Tensor, target_kv_len: torch.Tensor,
                                   draft_kv_len: Optional[torch.Tensor] = None, correction_processed: bool = True,
                                   history: Optional[torch.Tensor] = None,
                                   committed_len: Optional[torch.Tensor] = None,
                                   path_nodes: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                   workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_tree_greedy and spec_commit_kv_lengths (gmax = nmax) of the same round, fused."""
    B = target_logits.shape[0]
    args, _ = _tree_args(target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted, path_nodes,
                         status, workspace)
    _check(load_library().spec_verify_tree_greedy_commit(
        *args, *_commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len),
        _stream(stream)))


def prepare_verify_tree_greedy_commit(target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted,
                                      target_kv_len, draft_kv_len=None, correction_processed=True, history=None,
                                      committed_len=None, path_nodes=None, status=None, workspace=None,
                                      stream=None) -> "_Prepared":
    B = target_logits.shape[0]
    args, ws = _tree_args(target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted, path_nodes,
                          status, workspace)
    args = args + _commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len) + \
        (_stream(stream),)
    keep = (target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted, path_nodes, status, ws,
            target_kv_len, draft_kv_len, history, committed_len)
    return _Prepared(load_library().spec_verify_tree_greedy_commit, args, keep)


def prepare_verify_tree_greedy(target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted,
                               path_nodes=None, status=None, workspace=None, stream=None) -> "_Prepared":
    B, np1, V = target_logits.shape
    nmax = np1 - 1
    lib = load_library()
    ws, wsp, wsn = _ws(workspace, B, nmax, V, _dtype_code(target_logits), target_logits.device)
    args = (_ptr(target_logits, "target_logits"), _dtype_code(target_logits),
            _ptr(node_tokens, "node_tokens", torch.int32, (B, nmax)),
            _ptr(node_parents, "node_parents", torch.int32, (B, nmax)),
            _ptr(num_nodes, "num_nodes", torch.int32, (B,)), B, nmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, nmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(path_nodes, "path_nodes", torch.int32, (B, nmax)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream))
    keep = (target_logits, node_tokens, node_parents, num_nodes, out_tokens, num_accepted, path_nodes, status, ws)
    return _Prepared(lib.spec_verify_tree_greedy, args, keep)


def _split_shapes(saved_logits, block_logits):
    B, V = saved_logits.shape
    if block_logits is None:
        return B, 0, V
    Bb, gmax, Vb = block_logits.shape
    if (Bb, Vb) != (B, V) or block_logits.dtype != saved_logits.dtype:
        raise ValueError(f"block_logits {tuple(block_logits.shape)} does not match saved_logits {(B, V)}")
    return B, gmax, V


def spec_verify_greedy_split(saved_logits: torch.Tensor, block_logits: Optional[torch.Tensor],
                             draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                             out_tokens: torch.Tensor, num_accepted: torch.Tensor,
                             status: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_greedy with target row 0 (saved_logits [B][V]) apart from rows 1..gmax
    (block_logits [B][gmax][V])."""
    B, gmax, V = _split_shapes(saved_logits, block_logits)
    lib = load_library()
    code = _dtype_code(saved_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, saved_logits.device)
    _check(lib.spec_verify_greedy_split(
        _ptr(saved_logits, "saved_logits"), _ptr(block_logits, "block_logits"), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def spec_verify_sample_split(saved_logits: torch.Tensor, block_logits: Optional[torch.Tensor],
                             draft_logits: torch.Tensor, draft_tokens: torch.Tensor,
                             num_draft: Optional[torch.Tensor], temperature: torch.Tensor,
                             u_accept: torch.Tensor, u_sample: torch.Tensor, out_tokens: torch.Tensor,
                             num_accepted: torch.Tensor, diag: Optional[torch.Tensor] = None,
                             status: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample with target row 0 (saved_logits [B][V]) apart from rows 1..gmax
    (block_logits [B][gmax][V])."""
    B, gmax, V = _split_shapes(saved_logits, block_logits)
    if draft_logits.dtype != saved_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    lib = load_library()
    code = _dtype_code(saved_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, saved_logits.device)
    _check(lib.spec_verify_sample_split(
        _ptr(saved_logits, "saved_logits"), _ptr(block_logits, "block_logits"),
        _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)),
        _ptr(temperature, "temperature", torch.float32, (B,)),
        _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
        _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
        _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream)))


def spec_verify_sample_static(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                              draft_tokens: torch.Tensor, num_draft: Optional[torch.Tensor],
                              temperature: torch.Tensor, u_accept: torch.Tensor,
                              u_sample: torch.Tensor, out_tokens: torch.Tensor,
                              num_accepted: torch.Tensor, diag: Optional[torch.Tensor] = None,
                              status: Optional[torch.Tensor] = None, stream=None) -> None:
    """spec_verify_sample on the library's per-device static workspace: allocates nothing.
    Calls on one device share that workspace, so calls that may overlap must be serialised;
    the first call on a device clears it and should come before any stream capture."""
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    lib = load_library()
    code = _dtype_code(target_logits)
    _check(lib.spec_verify_sample_static(
        _ptr(target_logits, "target_logits"),
        _ptr(draft_logits, "draft_logits", None, (B, gmax, V)), code,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
        _ptr(num_draft, "num_draft", torch.int32, (B,)),
        _ptr(temperature, "temperature", torch.float32, (B,)),
        _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
        _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
        _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
        _ptr(status, "status", torch.int32, (B,)), _stream(stream)))


def spec_apply_stops(out_tokens: torch.Tensor, num_accepted: torch.Tensor, eos_id: int,
                     max_new: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    """Cut each round's emit at its first end token and to the remaining budget, in place."""
    B, gp1 = out_tokens.shape
    lib = load_library()
    _check(lib.spec_apply_stops(
        _ptr(out_tokens, "out_tokens", torch.int32, (B, gp1)),
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)), B, gp1 - 1, int(eos_id),
        _ptr(max_new, "max_new", torch.int32, (B,)),
        _ptr(status, "status", torch.int32, (B,)), _stream(stream)))


def _commit_gmax(out_tokens, gmax):
    if out_tokens is not None:
        g = out_tokens.shape[1] - 1
        if gmax is not None and gmax != g:
            raise ValueError(f"gmax={gmax} disagrees with out_tokens width {g + 1}")
        return g
    if gmax is None:
        raise ValueError("gmax is required when out_tokens is not given")
    return int(gmax)


def spec_commit_kv_lengths(num_accepted: torch.Tensor, target_kv_len: torch.Tensor,
                           draft_kv_len: Optional[torch.Tensor], correction_processed: bool,
                           out_tokens: Optional[torch.Tensor] = None,
                           history: Optional[torch.Tensor] = None,
                           committed_len: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None,
                           gmax: Optional[int] = None) -> None:
    B = num_accepted.shape[0]
    gmax = _commit_gmax(out_tokens, gmax)
    cap = history.shape[1] if history is not None else 0
    lib = load_library()
    _check(lib.spec_commit_kv_lengths(
        _ptr(num_accepted, "num_accepted", torch.int32, (B,)), B,
        _ptr(target_kv_len, "target_kv_len", torch.int32, (B,)),
        _ptr(draft_kv_len, "draft_kv_len", torch.int32, (B,)), int(bool(correction_processed)),
        _ptr(out_tokens, "out_tokens", torch.int32), gmax,
        _ptr(history, "history", torch.int32), _ptr(committed_len, "committed_len", torch.int32, (B,)),
        cap, _ptr(status, "status", torch.int32, (B,)), _stream(stream)))


def spec_launch_count() -> int:
    return int(load_library().spec_launch_count())


def spec_verify_plan(V: int, dtype: int = SPEC_BF16):
    """(blocks per sequence, vocabulary ids per block) a verify call uses for this V."""
    cl, ch = ctypes.c_int(), ctypes.c_int()
    _check(load_library().spec_verify_plan(V, dtype, ctypes.byref(cl), ctypes.byref(ch)))
    return cl.value, ch.value


class _Prepared:
    """A verify/commit call whose arguments were checked and marshalled once; calling it
    re-issues the same C call (same buffers, same stream) with no per-call Python checks."""

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self):
        _check(self._fn(*self._args))


def prepare_verify_sample(target_logits, draft_logits, draft_tokens, num_draft, temperature,
                          u_accept, u_sample, out_tokens, num_accepted, diag=None, status=None,
                          workspace=None, stream=None) -> _Prepared:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    lib = load_library()
    ws, wsp, wsn = _ws(workspace, B, gmax, V, _dtype_code(target_logits), target_logits.device)
    args = (_ptr(target_logits, "target_logits"),
            _ptr(draft_logits, "draft_logits", target_logits.dtype, (B, gmax, V)),
            _dtype_code(target_logits),
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)),
            _ptr(temperature, "temperature", torch.float32, (B,)),
            _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
            _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream))
    keep = (target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept,
            u_sample, out_tokens, num_accepted, diag, status, ws)
    return _Prepared(lib.spec_verify_sample, args, keep)


def prepare_verify_greedy_commit(target_logits, draft_tokens, num_draft, out_tokens, num_accepted, target_kv_len,
                                 draft_kv_len=None, correction_processed=True, history=None, committed_len=None,
                                 status=None, workspace=None, stream=None) -> _Prepared:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    code = _dtype_code(target_logits)
    ws, wsp, wsn = _ws(workspace, B, gmax, V, code, target_logits.device)
    args = (_ptr(target_logits, "target_logits"), code,
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn,
            *_commit_args(B, target_kv_len, draft_kv_len, correction_processed, history, committed_len),
            _stream(stream))
    keep = (target_logits, draft_tokens, num_draft, out_tokens, num_accepted, status, ws, target_kv_len,
            draft_kv_len, history, committed_len)
    return _Prepared(load_library().spec_verify_greedy_commit, args, keep)


def prepare_verify_sample_commit(target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept,
                                 u_sample, out_tokens, num_accepted, target_kv_len, draft_kv_len=None,
                                 correction_processed=True, history=None, committed_len=None, diag=None,
                                 status=None, workspace=None, stream=None) -> _Prepared:
    args, ws = _sample_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept,
                                   u_sample, out_tokens, num_accepted, diag, status, workspace, target_kv_len,
                                   draft_kv_len, correction_processed, history, committed_len, stream)
    keep = (target_logits, draft_logits, draft_tokens, num_draft, temperature, u_accept, u_sample, out_tokens,
            num_accepted, diag, status, ws, target_kv_len, draft_kv_len, history, committed_len)
    return _Prepared(load_library().spec_verify_sample_commit, args, keep)


def prepare_verify_sample_truncated(target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k,
                                    top_p, u_accept, u_sample, out_tokens, num_accepted, diag=None, status=None,
                                    workspace=None, stream=None) -> _Prepared:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    lib = load_library()
    ws, wsp, wsn = _ws(workspace, B, gmax, V, _dtype_code(target_logits), target_logits.device)
    args = (_ptr(target_logits, "target_logits"),
            _ptr(draft_logits, "draft_logits", target_logits.dtype, (B, gmax, V)),
            _dtype_code(target_logits),
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)),
            _ptr(temperature, "temperature", torch.float32, (B,)),
            _ptr(top_k, "top_k", torch.int32, (B,)), _ptr(top_p, "top_p", torch.float32, (B,)),
            _ptr(u_accept, "u_accept", torch.float32, (B, gmax)),
            _ptr(u_sample, "u_sample", torch.float32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(diag, "diag", torch.float32, (B, 2 * gmax + 1)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream))
    keep = (target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k, top_p, u_accept,
            u_sample, out_tokens, num_accepted, diag, status, ws)
    return _Prepared(lib.spec_verify_sample_truncated, args, keep)


def prepare_verify_sample_truncated_commit(target_logits, draft_logits, draft_tokens, num_draft, temperature,
                                           top_k, top_p, u_accept, u_sample, out_tokens, num_accepted,
                                           target_kv_len, draft_kv_len=None, correction_processed=True,
                                           history=None, committed_len=None, diag=None, status=None,
                                           workspace=None, stream=None) -> _Prepared:
    args, ws = _truncated_commit_args(target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k,
                                      top_p, u_accept, u_sample, out_tokens, num_accepted, diag, status, workspace,
                                      target_kv_len, draft_kv_len, correction_processed, history, committed_len,
                                      stream)
    keep = (target_logits, draft_logits, draft_tokens, num_draft, temperature, top_k, top_p, u_accept, u_sample,
            out_tokens, num_accepted, diag, status, ws, target_kv_len, draft_kv_len, history, committed_len)
    return _Prepared(load_library().spec_verify_sample_truncated_commit, args, keep)


def prepare_verify_greedy(target_logits, draft_tokens, num_draft, out_tokens, num_accepted,
                          status=None, workspace=None, stream=None) -> _Prepared:
    B, gp1, V = target_logits.shape
    gmax = gp1 - 1
    lib = load_library()
    ws, wsp, wsn = _ws(workspace, B, gmax, V, _dtype_code(target_logits), target_logits.device)
    args = (_ptr(target_logits, "target_logits"), _dtype_code(target_logits),
            _ptr(draft_tokens, "draft_tokens", torch.int32, (B, gmax)),
            _ptr(num_draft, "num_draft", torch.int32, (B,)), B, gmax, V,
            _ptr(out_tokens, "out_tokens", torch.int32, (B, gmax + 1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)),
            _ptr(status, "status", torch.int32, (B,)), wsp, wsn, _stream(stream))
    keep = (target_logits, draft_tokens, num_draft, out_tokens, num_accepted, status, ws)
    return _Prepared(lib.spec_verify_greedy, args, keep)


def prepare_apply_stops(out_tokens, num_accepted, eos_id, max_new=None, status=None, stream=None) -> _Prepared:
    B, gp1 = out_tokens.shape
    lib = load_library()
    args = (_ptr(out_tokens, "out_tokens", torch.int32, (B, gp1)),
            _ptr(num_accepted, "num_accepted", torch.int32, (B,)), B, gp1 - 1, int(eos_id),
            _ptr(max_new, "max_new", torch.int32, (B,)), _ptr(status, "status", torch.int32, (B,)),
            _stream(stream))
    return _Prepared(lib.spec_apply_stops, args, (out_tokens, num_accepted, max_new, status))


def prepare_commit_kv_lengths(num_accepted, target_kv_len, draft_kv_len, correction_processed,
                              out_tokens=None, history=None, committed_len=None, status=None,
                              stream=None, gmax=None) -> _Prepared:
    B = num_accepted.shape[0]
    gmax = _commit_gmax(out_tokens, gmax)
    cap = history.shape[1] if history is not None else 0
    lib = load_library()
    args = (_ptr(num_accepted, "num_accepted", torch.int32, (B,)), B,
            _ptr(target_kv_len, "target_kv_len", torch.int32, (B,)),
            _ptr(draft_kv_len, "draft_kv_len", torch.int32, (B,)), int(bool(correction_processed)),
            _ptr(out_tokens, "out_tokens", torch.int32), gmax, _ptr(history, "history", torch.int32),
            _ptr(committed_len, "committed_len", torch.int32, (B,)), cap,
            _ptr(status, "status", torch.int32, (B,)), _stream(stream))
    keep = (num_accepted, target_kv_len, draft_kv_len, out_tokens, history, committed_len, status)
    return _Prepared(lib.spec_commit_kv_lengths, args, keep)
