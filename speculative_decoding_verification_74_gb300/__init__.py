"""Python binding of libsv: speculative-decoding draft verification and D-cut depth scheduling
on GB300 (sm_103a).

This module only marshals arguments: every step of verification and scheduling runs in the
CUDA kernels of ``libsv.so`` (built in-tree by ``build.build()``).  PyTorch supplies device
memory and streams.  There is no CPU fallback: if the library is missing or cannot be loaded,
every call raises.

The ``sv_*`` functions mirror the C ABI in ``include/sv.h`` one to one (tensors in place of
pointers, ``None`` for NULL).  The lower-case helpers (``verify_greedy``, ``verify_sample``,
``verify_ragged``, ``schedule_depth``) derive sizes and strides from the tensors and allocate
outputs and workspaces.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsv.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "sv.h")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_WORKSPACE, SV_ERR_CUDA, SV_ERR_DEVICE_INPUT, SV_ERR_TIMEOUT = range(6)
SV_BF16, SV_F32 = 0, 1
SV_OP_VERIFY, SV_OP_SCHEDULE, SV_OP_TREE = 0, 1, 2
SV_OBJ_THROUGHPUT, SV_OBJ_NET = 0, 1
SV_PHASE_STATS, SV_PHASE_ACCEPT, SV_PHASE_WEIGHTS, SV_PHASE_PICK = range(4)
(SV_DEV_BAD_TOKEN, SV_DEV_BAD_TEMPERATURE, SV_DEV_BAD_KEEP_LEN, SV_DEV_BAD_OFFSETS, SV_DEV_NO_DRAFT_ROWS,
 SV_DEV_BAD_ALPHA, SV_DEV_BAD_DRAFT_LEN, SV_DEV_TIMEOUT, SV_DEV_BAD_PARENT) = (1 << b for b in range(9))
SV_FLAG_Q_ZERO, SV_FLAG_Z_ZERO, SV_FLAG_INVALID = 1, 2, 4
(SV_KERNEL_ROW_STATS, SV_KERNEL_COMBINE, SV_KERNEL_SCHEDULE, SV_KERNEL_MASS, SV_KERNEL_PICK, SV_KERNEL_TREE_WALK,
 SV_NUM_KERNELS) = range(7)
KERNEL_NAMES = ("row_stats", "combine", "schedule", "mass", "pick", "tree_walk")

_c = ctypes
_vp, _i32, _i64, _u32, _u64, _f32, _sz = (_c.c_void_p, _c.c_int32, _c.c_int64, _c.c_uint32, _c.c_uint64,
                                         _c.c_float, _c.c_size_t)

_SIGS = {
    "sv_abi_version": (_c.c_int, []),
    "sv_workspace_size": (_sz, [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int]),
    "sv_verify_greedy": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                    _vp, _vp, _vp, _sz, _vp]),
    "sv_verify_sample": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _vp, _u64, _u32, _vp, _c.c_int, _c.c_int,
                                    _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sv_verify_ragged": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _c.c_int, _vp, _vp,
                                    _u64, _u32, _vp, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _sz, _vp]),
    "sv_verify_sample_noalloc": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _vp, _u64, _u32, _vp, _c.c_int,
                                            _c.c_int, _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp, _vp]),
    "sv_schedule_depth": (_c.c_int, [_vp, _c.c_int, _vp, _c.c_int, _c.c_int, _f32, _f32, _c.c_int, _vp,
                                     _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sv_schedule_depth_table": (_c.c_int, [_vp, _c.c_int, _vp, _c.c_int, _c.c_int, _vp, _vp, _c.c_int,
                                           _c.c_int, _vp, _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp, _sz,
                                           _vp]),
    "sv_verify_tree": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _u64, _u32, _vp, _c.c_int,
                                  _c.c_int, _c.c_int, _c.c_int, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sv_vocab_chunks": (_c.c_int, [_c.c_int, _c.c_int, _c.POINTER(_c.c_int), _c.POINTER(_c.c_int)]),
    "sv_verify_regions": (_c.c_int, [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.POINTER(_sz), _c.POINTER(_sz),
                                     _c.POINTER(_sz), _c.POINTER(_sz), _c.POINTER(_sz)]),
    "sv_verify_sample_phase": (_c.c_int, [_vp, _i64, _vp, _i64, _vp, _vp, _u64, _u32, _vp, _c.c_int, _c.c_int,
                                          _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _vp, _vp, _vp, _vp,
                                          _vp, _vp, _sz, _vp]),
    "sv_test_stall_next_verify": (None, [_c.c_int]),
    "sv_query_status": (_c.c_int, [_vp, _vp, _c.POINTER(_u32)]),
    "sv_status_string": (_c.c_char_p, [_c.c_int]),
    "sv_last_error_string": (_c.c_char_p, []),
    "sv_profile_enable": (None, [_c.c_int]),
    "sv_profile_collect": (_c.c_int, [_c.POINTER(_c.c_double), _c.POINTER(_i64)]),
    "sv_profile_reset": (None, []),
    "sv_launch_count": (_i64, []),
}

_lib = None


class SVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libsv status {status}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libsv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Function names declared in include/sv.h."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(sv_\w+)\s*\(", txt, re.M)))


def _check(status: int) -> None:
    if status != SV_OK:
        L = lib()
        raise SVError(status, L.sv_last_error_string().decode() or L.sv_status_string(status).decode())


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libsv takes device tensors")
    return t.data_ptr()


def _need(t, name: str, dtype, count: int = 0) -> None:
    """Host check of one array argument before its pointer reaches the kernels: its dtype, and
    at least `count` elements of its storage from its data pointer on (the kernels index past
    a view's shape when a stride says so).  Raw integer pointers are the caller's affair."""
    if t is None or isinstance(t, int):
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if count > 0:
        avail = t.untyped_storage().nbytes() // t.element_size() - t.storage_offset()
        if avail < count:
            raise ValueError(f"{name} holds {avail} elements from its data pointer, the call reads {count}")


def _logit_dtype(dt: int):
    return {SV_BF16: torch.bfloat16, SV_F32: torch.float32}.get(dt)


def _need_rows(t, name: str, dt: int, rows: int, stride: int, V: int) -> None:
    """Logit rows: rows x V elements at the given row stride."""
    _need(t, name, _logit_dtype(dt), (rows - 1) * stride + V if rows > 0 and stride >= V > 0 else 0)


def _ws_bytes(ws) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


# ------------------------------------------------------------------------------------------
# one-to-one C ABI (tensors for pointers, None for NULL); each raises SVError on failure
# ------------------------------------------------------------------------------------------

def sv_workspace_size(op: int, B: int, Kmax: int, V: int, dt: int) -> int:
    return int(lib().sv_workspace_size(op, B, Kmax, V, dt))


def sv_verify_greedy(target, t_row_stride, draft, d_row_stride, draft_tokens, dt, B, K, V, out_tokens,
                     out_accept_len, ws, stream=None) -> None:
    if B > 0 and K >= 0:
        _need_rows(target, "target", dt, B * (K + 1), t_row_stride, V)
        _need_rows(draft, "draft", dt, B * K, d_row_stride, V)
        _need(draft_tokens, "draft_tokens", torch.int32, B * K)
        _need(out_tokens, "out_tokens", torch.int32, B * (K + 1))
        _need(out_accept_len, "out_accept_len", torch.int32, B)
    _check(lib().sv_verify_greedy(_p(target), t_row_stride, _p(draft), d_row_stride, _p(draft_tokens), dt, B,
                                  K, V, _p(out_tokens), _p(out_accept_len), _p(ws),
                                  _ws_bytes(ws), _stream(stream)))


def sv_verify_sample(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round_,
                     request_ids, dt, B, K, V, out_tokens, out_accept_len, out_p, out_q, out_flags, ws,
                     stream=None) -> None:
    if B > 0 and K >= 0:
        _need_rows(target, "target", dt, B * (K + 1), t_row_stride, V)
        _need_rows(draft, "draft", dt, B * K, d_row_stride, V)
        _need(draft_tokens, "draft_tokens", torch.int32, B * K)
        _need(temperature, "temperature", torch.float32, B)
        _need(request_ids, "request_ids", torch.int32, B)
        _need(out_tokens, "out_tokens", torch.int32, B * (K + 1))
        _need(out_accept_len, "out_accept_len", torch.int32, B)
        _need(out_p, "out_p", torch.float32, B * K)
        _need(out_q, "out_q", torch.float32, B * K)
        _need(out_flags, "out_flags", torch.uint8, B)
    _check(lib().sv_verify_sample(_p(target), t_row_stride, _p(draft), d_row_stride, _p(draft_tokens),
                                  _p(temperature), seed & (2 ** 64 - 1), round_, _p(request_ids), dt, B, K, V,
                                  _p(out_tokens), _p(out_accept_len), _p(out_p), _p(out_q), _p(out_flags),
                                  _p(ws), _ws_bytes(ws), _stream(stream)))


def sv_verify_ragged(target, t_row_stride, t_row_offsets, t_rows, draft, d_row_stride, d_row_offsets, d_rows,
                     draft_tokens, tok_stride, keep_len, temperature, seed, round_, request_ids, dt, B, Kmax, V,
                     out_tokens, out_accept_len, out_p, out_q, out_flags, ws, stream=None) -> None:
    if B > 0 and Kmax >= 0:
        # the packed arrays hold t_rows / d_rows rows; the kernels bound every request's rows by them
        _need_rows(target, "target", dt, t_rows, t_row_stride, V)
        if draft is not None:
            _need_rows(draft, "draft", dt, d_rows, d_row_stride, V)
        _need(t_row_offsets, "t_row_offsets", torch.int32, B + 1)
        _need(d_row_offsets, "d_row_offsets", torch.int32, B + 1)
        _need(draft_tokens, "draft_tokens", torch.int32,
              (B - 1) * tok_stride + Kmax if Kmax > 0 and tok_stride >= Kmax else 0)
        _need(keep_len, "keep_len", torch.int32, B)
        _need(temperature, "temperature", torch.float32, B)
        _need(request_ids, "request_ids", torch.int32, B)
        _need(out_tokens, "out_tokens", torch.int32, B * (Kmax + 1))
        _need(out_accept_len, "out_accept_len", torch.int32, B)
        _need(out_p, "out_p", torch.float32, B * Kmax)
        _need(out_q, "out_q", torch.float32, B * Kmax)
        _need(out_flags, "out_flags", torch.uint8, B)
    _check(lib().sv_verify_ragged(_p(target), t_row_stride, _p(t_row_offsets), t_rows, _p(draft), d_row_stride,
                                  _p(d_row_offsets), d_rows, _p(draft_tokens), tok_stride, _p(keep_len),
                                  _p(temperature), seed & (2 ** 64 - 1), round_, _p(request_ids), dt, B, Kmax,
                                  V, _p(out_tokens), _p(out_accept_len), _p(out_p), _p(out_q), _p(out_flags),
                                  _p(ws), _ws_bytes(ws), _stream(stream)))


def sv_verify_sample_noalloc(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round_,
                             request_ids, dt, B, K, V, out_tokens, out_accept_len, out_p, out_q, out_flags,
                             stream=None) -> None:
    """sv_verify_sample on the library's built-in scratch (no workspace argument)."""
    if B > 0 and K >= 0:
        _need_rows(target, "target", dt, B * (K + 1), t_row_stride, V)
        _need_rows(draft, "draft", dt, B * K, d_row_stride, V)
        _need(draft_tokens, "draft_tokens", torch.int32, B * K)
        _need(temperature, "temperature", torch.float32, B)
        _need(request_ids, "request_ids", torch.int32, B)
        _need(out_tokens, "out_tokens", torch.int32, B * (K + 1))
        _need(out_accept_len, "out_accept_len", torch.int32, B)
        _need(out_p, "out_p", torch.float32, B * K)
        _need(out_q, "out_q", torch.float32, B * K)
        _need(out_flags, "out_flags", torch.uint8, B)
    _check(lib().sv_verify_sample_noalloc(_p(target), t_row_stride, _p(draft), d_row_stride, _p(draft_tokens),
                                          _p(temperature), seed & (2 ** 64 - 1), round_, _p(request_ids), dt, B,
                                          K, V, _p(out_tokens), _p(out_accept_len), _p(out_p), _p(out_q),
                                          _p(out_flags), _stream(stream)))


def sv_schedule_depth(alpha, alpha_stride, draft_len, B, Dmax, cost_a, cost_b, budget, ratios, objective,
                      out_keep_len, out_row_offsets, out_total_K, out_utility_q48, ws, stream=None) -> None:
    if B > 0 and Dmax >= 0:
        _need(alpha, "alpha", torch.float32, (B - 1) * alpha_stride + Dmax if Dmax > 0 and alpha_stride >= Dmax else 0)
        _need(draft_len, "draft_len", torch.int32, B)
        _need(out_keep_len, "out_keep_len", torch.int32, B)
        _need(out_row_offsets, "out_row_offsets", torch.int32, B + 1)
        _need(out_total_K, "out_total_K", torch.int32, 1)
        _need(out_utility_q48, "out_utility_q48", torch.int64, 1)
    rat = None
    n = 0
    if ratios is not None:
        n = len(ratios)
        rat = (ctypes.c_float * n)(*[float(r) for r in ratios])
    _check(lib().sv_schedule_depth(_p(alpha), alpha_stride, _p(draft_len), B, Dmax, float(cost_a),
                                   float(cost_b), budget, ctypes.cast(rat, ctypes.c_void_p) if rat else None,
                                   n, objective, _p(out_keep_len), _p(out_row_offsets), _p(out_total_K),
                                   _p(out_utility_q48), _p(ws), _ws_bytes(ws),
                                   _stream(stream)))


def sv_schedule_depth_table(alpha, alpha_stride, draft_len, B, Dmax, cost_K, cost_c, budget, ratios, objective,
                            out_keep_len, out_row_offsets, out_total_K, out_utility_q48, ws, stream=None) -> None:
    if B > 0 and Dmax >= 0:
        _need(alpha, "alpha", torch.float32, (B - 1) * alpha_stride + Dmax if Dmax > 0 and alpha_stride >= Dmax else 0)
        _need(draft_len, "draft_len", torch.int32, B)
        _need(out_keep_len, "out_keep_len", torch.int32, B)
        _need(out_row_offsets, "out_row_offsets", torch.int32, B + 1)
        _need(out_total_K, "out_total_K", torch.int32, 1)
        _need(out_utility_q48, "out_utility_q48", torch.int64, 1)
    rat = None
    n = 0
    if ratios is not None:
        n = len(ratios)
        rat = (ctypes.c_float * n)(*[float(r) for r in ratios])
    nk = len(cost_K)
    if len(cost_c) != nk:
        raise SVError(SV_ERR_INVALID_ARG, "cost_K and cost_c differ in length")
    ks = (ctypes.c_int32 * max(nk, 1))(*[int(k) for k in cost_K])
    cs = (ctypes.c_double * max(nk, 1))(*[float(c) for c in cost_c])
    _check(lib().sv_schedule_depth_table(_p(alpha), alpha_stride, _p(draft_len), B, Dmax,
                                         ctypes.cast(ks, ctypes.c_void_p), ctypes.cast(cs, ctypes.c_void_p), nk,
                                         budget, ctypes.cast(rat, ctypes.c_void_p) if rat else None, n, objective,
                                         _p(out_keep_len), _p(out_row_offsets), _p(out_total_K),
                                         _p(out_utility_q48), _p(ws), _ws_bytes(ws),
                                         _stream(stream)))


def sv_verify_tree(target, t_row_stride, draft, d_row_stride, node_offsets, n_rows, parent, tokens, temperature,
                   seed, round_, request_ids, dt, B, Nmax, V, out_path, out_tokens, out_accept_len, out_flags, ws,
                   stream=None) -> None:
    if B > 0:
        # the packed arrays hold n_rows rows; the kernels bound every request's rows by it
        _need_rows(target, "target", dt, n_rows, t_row_stride, V)
        if draft is not None:
            _need_rows(draft, "draft", dt, n_rows, d_row_stride, V)
        _need(node_offsets, "node_offsets", torch.int32, B + 1)
        _need(parent, "parent", torch.int32, n_rows)
        _need(tokens, "tokens", torch.int32, n_rows)
        _need(temperature, "temperature", torch.float32, B)
        _need(request_ids, "request_ids", torch.int32, B)
        _need(out_path, "out_path", torch.int32, B * Nmax)
        _need(out_tokens, "out_tokens", torch.int32, B * Nmax)
        _need(out_accept_len, "out_accept_len", torch.int32, B)
        _need(out_flags, "out_flags", torch.uint8, B)
    _check(lib().sv_verify_tree(_p(target), t_row_stride, _p(draft), d_row_stride, _p(node_offsets), n_rows,
                                _p(parent), _p(tokens), _p(temperature), seed & (2 ** 64 - 1), round_,
                                _p(request_ids), dt, B, Nmax, V, _p(out_path), _p(out_tokens), _p(out_accept_len),
                                _p(out_flags), _p(ws), _ws_bytes(ws), _stream(stream)))


def sv_vocab_chunks(V: int, dt: int) -> tuple[int, int]:
    cl, nc = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().sv_vocab_chunks(V, dt, ctypes.byref(cl), ctypes.byref(nc)))
    return cl.value, nc.value


def sv_verify_regions(B: int, K: int, V: int, dt: int) -> dict:
    """Workspace byte offsets and sizes of the chunk records and the two range-sum arrays."""
    v = [ctypes.c_size_t(0) for _ in range(5)]
    _check(lib().sv_verify_regions(B, K, V, dt, *(ctypes.byref(x) for x in v)))
    return {"rec_offset": v[0].value, "rec_bytes": v[1].value, "mass_offset": v[2].value,
            "mass_p_offset": v[3].value, "mass_bytes": v[4].value}


def sv_verify_sample_phase(target, t_row_stride, draft, d_row_stride, draft_tokens, temperature, seed, round_,
                           request_ids, dt, B, K, V, c_begin, c_end, phase, out_tokens, out_accept_len, out_p,
                           out_q, out_flags, ws, stream=None) -> None:
    if B > 0 and K >= 0:
        # the arrays hold the shard's columns: those of chunks [c_begin, c_end)
        cl, nc = sv_vocab_chunks(V, dt)
        v_local = min(V, c_end * cl) - c_begin * cl if 0 <= c_begin < c_end <= nc else 0
        _need_rows(target, "target", dt, B * (K + 1), t_row_stride, v_local)
        _need_rows(draft, "draft", dt, B * K, d_row_stride, v_local)
        _need(draft_tokens, "draft_tokens", torch.int32, B * K)
        _need(temperature, "temperature", torch.float32, B)
        _need(request_ids, "request_ids", torch.int32, B)
        _need(out_tokens, "out_tokens", torch.int32, B * (K + 1))
        _need(out_accept_len, "out_accept_len", torch.int32, B)
        _need(out_p, "out_p", torch.float32, B * K)
        _need(out_q, "out_q", torch.float32, B * K)
        _need(out_flags, "out_flags", torch.uint8, B)
    _check(lib().sv_verify_sample_phase(_p(target), t_row_stride, _p(draft), d_row_stride, _p(draft_tokens),
                                        _p(temperature), seed & (2 ** 64 - 1), round_, _p(request_ids), dt, B, K, V,
                                        c_begin, c_end, phase, _p(out_tokens), _p(out_accept_len), _p(out_p),
                                        _p(out_q), _p(out_flags), _p(ws), _ws_bytes(ws), _stream(stream)))


def sv_test_stall_next_verify(wait_limit_ms: int) -> None:
    lib().sv_test_stall_next_verify(int(wait_limit_ms))


def sv_query_status(ws, stream=None) -> tuple[int, int]:
    v = ctypes.c_uint32(0)
    st = lib().sv_query_status(_p(ws), _stream(stream), ctypes.byref(v))
    if st not in (SV_OK, SV_ERR_DEVICE_INPUT, SV_ERR_TIMEOUT):
        _check(st)
    return st, int(v.value)


def sv_profile_enable(on: bool) -> None:
    lib().sv_profile_enable(1 if on else 0)


def sv_profile_collect() -> tuple[list[float], list[int]]:
    ms = (ctypes.c_double * SV_NUM_KERNELS)()
    n = (ctypes.c_int64 * SV_NUM_KERNELS)()
    _check(lib().sv_profile_collect(ms, n))
    return list(ms), list(n)


def sv_profile_reset() -> None:
    lib().sv_profile_reset()


def sv_launch_count() -> int:
    return int(lib().sv_launch_count())


# ------------------------------------------------------------------------------------------
# convenience wrappers
# ------------------------------------------------------------------------------------------

def workspace(op: int, B: int, Kmax: int, V: int, dt: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (torch allocations are 512-byte aligned)."""
    n = sv_workspace_size(op, B, Kmax, V, dt)
    if n == 0:
        raise ValueError("invalid sizes for sv_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _rows(x: torch.Tensor):
    """(base tensor, row stride) for [..., V] logits with a contiguous last dimension."""
    if x.numel() == 0:
        return x, x.shape[-1]
    if x.stride(-1) != 1:
        raise ValueError("logit rows must be contiguous")
    return x, (x.stride(-2) if x.dim() >= 2 else x.shape[-1])


def num_rows(x: torch.Tensor) -> int:
    """Rows of V logits in a [..., V] tensor."""
    return x.numel() // x.shape[-1] if x.shape[-1] > 0 else 0


def verify_greedy(target, K, *, draft=None, draft_tokens=None, ws=None, stream=None):
    """target [B*(K+1), V] (or [B, K+1, V]); draft [B*K, V] or draft_tokens [B, K]."""
    V = target.shape[-1]
    B = target.numel() // V // (K + 1)
    dt = _dt(target)
    _, ts = _rows(target)
    ds = _rows(draft)[1] if draft is not None else V
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=target.device)
    out_len = torch.empty(B, dtype=torch.int32, device=target.device)
    if ws is None:
        ws = workspace(SV_OP_VERIFY, B, K, V, dt, target.device)
    sv_verify_greedy(target, ts, draft, ds, draft_tokens, dt, B, K, V, out_tok, out_len, ws, stream)
    return out_tok, out_len


def verify_sample(target, draft, draft_tokens, temperature, K, *, seed=0, round_=0, request_ids=None,
                  ws=None, stream=None, want_pq=True):
    V = target.shape[-1]
    B = target.numel() // V // (K + 1)
    dt = _dt(target)
    dev = target.device
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    out_p = torch.empty((B, K), dtype=torch.float32, device=dev) if want_pq else None
    out_q = torch.empty((B, K), dtype=torch.float32, device=dev) if want_pq else None
    out_f = torch.empty(B, dtype=torch.uint8, device=dev)
    if ws is None:
        ws = workspace(SV_OP_VERIFY, B, K, V, dt, dev)
    ds = _rows(draft)[1] if draft is not None else V
    sv_verify_sample(target, _rows(target)[1], draft, ds, draft_tokens, temperature, seed, round_, request_ids,
                     dt, B, K, V, out_tok, out_len, out_p, out_q, out_f, ws, stream)
    return out_tok, out_len, out_p, out_q, out_f


def verify_tree(target, draft, node_offsets, parent, tokens, temperature, Nmax, *, seed=0, round_=0,
                request_ids=None, ws=None, stream=None, out=None):
    """Token-tree verification.  target / draft [rows, V]: node c of request i is row
    node_offsets[i] + c; parent / tokens [rows] int32 per node; temperature [B].  Returns
    (path [B, Nmax], tokens [B, Nmax], accept_len [B], flags [B])."""
    V = target.shape[-1]
    B = node_offsets.numel() - 1
    dt = _dt(target)
    dev = target.device
    if out is None:
        out = (torch.empty((B, Nmax), dtype=torch.int32, device=dev),
               torch.empty((B, Nmax), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.uint8, device=dev))
    if ws is None:
        ws = workspace(SV_OP_TREE, B, Nmax, V, dt, dev)
    ds = _rows(draft)[1] if draft is not None else V
    sv_verify_tree(target, _rows(target)[1], draft, ds, node_offsets, num_rows(target), parent, tokens, temperature,
                   seed, round_, request_ids, dt, B, Nmax, V, *out, ws, stream)
    return out


def verify_ragged(target, t_row_offsets, draft, d_row_offsets, draft_tokens, keep_len, temperature, Kmax, *,
                  seed=0, round_=0, request_ids=None, ws=None, stream=None, want_pq=True, out=None):
    V = target.shape[-1]
    B = keep_len.numel()
    dt = _dt(target)
    dev = target.device
    if out is None:
        out = (torch.empty((B, Kmax + 1), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty((B, Kmax), dtype=torch.float32, device=dev) if want_pq else None,
               torch.empty((B, Kmax), dtype=torch.float32, device=dev) if want_pq else None,
               torch.empty(B, dtype=torch.uint8, device=dev))
    if ws is None:
        ws = workspace(SV_OP_VERIFY, B, Kmax, V, dt, dev)
    ds = _rows(draft)[1] if draft is not None else V
    ts_ = draft_tokens.stride(0) if draft_tokens is not None else Kmax
    sv_verify_ragged(target, _rows(target)[1], t_row_offsets, num_rows(target), draft, ds, d_row_offsets,
                     num_rows(draft) if draft is not None else 0, draft_tokens, ts_, keep_len, temperature, seed,
                     round_, request_ids, dt, B, Kmax, V, *out, ws, stream)
    return out


def schedule_depth(alpha, cost_a, cost_b, budget, *, draft_len=None, ratios=None, objective=SV_OBJ_THROUGHPUT,
                   ws=None, stream=None, out=None, cost_table=None):
    """alpha [B, Dmax] float32 (device).  Returns (keep_len [B], row_offsets [B+1], total_K [1], U_q48 [1]).
    cost_table = (token counts, latencies), e.g. from cost_table.profile_cost_table, replaces the linear
    cost cost_a + cost_b * K (sv_schedule_depth_table)."""
    B, Dmax = alpha.shape
    dev = alpha.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B + 1, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.int64, device=dev))
    if ws is None:
        ws = workspace(SV_OP_SCHEDULE, B, Dmax, 1, SV_F32, dev)
    if cost_table is not None:
        sv_schedule_depth_table(alpha, alpha.stride(0), draft_len, B, Dmax, cost_table[0], cost_table[1], budget,
                                ratios, objective, *out, ws, stream)
    else:
        sv_schedule_depth(alpha, alpha.stride(0), draft_len, B, Dmax, cost_a, cost_b, budget, ratios, objective,
                          *out, ws, stream)
    return out
