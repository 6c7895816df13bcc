"""Python binding of the BA-Att C-ABI library (``lib/libba.so``).

Argument marshalling only: tensors are passed as raw device pointers with the
current CUDA stream; every step of selection and attention runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no CPU fallback: if the library is missing or no GPU is present the calls
raise.

The names follow the C ABI (``include/ba.h``): ``ba_select``,
``ba_sparse_attn``, ``ba_attn_dense``.  Each has a ``*_into`` form that
writes caller-provided tensors and allocates nothing.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import _build

__all__ = ["load", "ba_select", "ba_select_into", "ba_select_noalloc_into", "ba_select_isolated",
           "ba_select_isolated_into", "ba_sparse_attn", "ba_sparse_attn_into", "ba_block_fidelity",
           "ba_active_tokens", "ba_reuse_rows",
           "ba_attn_dense", "ba_attn_dense_into", "ba_merge_lse", "ba_merge_lse_into",
           "last_device_error", "selftest_wait_timeout", "ba_validate_selection", "selftest_attn_stall", "BAError",
           "SORT_NONE", "SORT_K", "SORT_Q", "SORT_QK", "select_workspace_size",
           "sparse_attn_workspace_size", "header_functions", "LIB_PATH"]

SORT_NONE, SORT_K, SORT_Q, SORT_QK = 0, 1, 2, 3
LIB_PATH = _build.LIB_PATH
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ba.h")

_c_void_p, _c_int, _c_float, _c_size = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_c_u32p = ctypes.POINTER(ctypes.c_uint32)

_SIGS = {
    "ba_status_string": (ctypes.c_char_p, [_c_int]),
    "ba_version": (ctypes.c_char_p, []),
    "ba_select_workspace_size": (_c_size, [_c_int] * 8),
    "ba_select": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 6 + [_c_float, _c_int, _c_int]
                  + [_c_void_p] * 6 + [_c_size, _c_void_p]),
    "ba_sparse_attn_workspace_size": (_c_size, [_c_int] * 8),
    "ba_sparse_attn": (_c_int, [_c_void_p] * 3 + [_c_int] * 5 + [_c_void_p] * 3 + [_c_int, _c_float]
                       + [_c_void_p] * 3 + [_c_size, _c_void_p]),
    "ba_attn_dense": (_c_int, [_c_void_p] * 3 + [_c_int] * 4 + [_c_float] + [_c_void_p] * 3),
    "ba_last_device_error": (_c_int, [_c_void_p, _c_u32p]),
    "ba_selftest_wait_timeout": (_c_int, [ctypes.c_uint32, _c_void_p]),
    "ba_validate_selection": (_c_int, [_c_void_p] * 3 + [_c_int] * 5 + [_c_u32p, _c_void_p]),
    "ba_selftest_attn_stall": (_c_int, [_c_void_p] * 3 + [_c_int] * 4 + [ctypes.c_uint32] + [_c_void_p] * 3),
    "ba_merge_lse": (_c_int, [_c_void_p] * 4 + [ctypes.c_int64, _c_int] + [_c_void_p] * 3),
    "ba_select_isolated": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 8 + [_c_float, _c_int, _c_int]
                           + [_c_void_p] * 6 + [_c_size, _c_void_p]),
    "ba_block_fidelity_workspace_size": (_c_size, [_c_int] * 5),
    "ba_block_fidelity": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 5 + [_c_void_p] * 3 + [_c_float]
                          + [_c_void_p, _c_int] + [_c_void_p] * 5 + [_c_size, _c_void_p]),
    "ba_active_tokens": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 6 + [_c_void_p, _c_void_p, _c_void_p]),
    "ba_reuse_rows": (_c_int, [_c_void_p] * 3 + [ctypes.c_int64, _c_int] + [_c_void_p] * 3),
    "ba_select_noalloc": (_c_int, [_c_void_p, _c_void_p] + [_c_int] * 6 + [_c_float, _c_int, _c_int]
                          + [_c_void_p] * 5 + [_c_void_p]),
}

_lib = None


class BAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().ba_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg}")


def header_functions() -> list[str]:
    """Names of the functions declared in include/ba.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ba_[a-z_]+)\s*\(", text, flags=re.M)


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the shared library (building it first when it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libba.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class _on_device:
    """Makes a tensor's device current around a library call (the library
    launches on the current device and the caller's stream of that device)."""

    def __init__(self, t):
        self.ctx = _torch().cuda.device(t.device)

    def __enter__(self):
        self.ctx.__enter__()

    def __exit__(self, *exc):
        return self.ctx.__exit__(*exc)


def _check(status: int, where: str):
    if status != 0:
        raise BAError(status, where)


def _need_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("ba_*: every tensor must live on a CUDA device (no CPU path)")


def select_workspace_size(b, h, L, d, B, kappa, sort_mode=SORT_QK, sort_window=0) -> int:
    return int(load().ba_select_workspace_size(b, h, L, d, B, kappa, sort_mode, sort_window))


def sparse_attn_workspace_size(b, h, L, d, B, kappa, has_perm_q=True, has_perm_k=True) -> int:
    return int(load().ba_sparse_attn_workspace_size(b, h, L, d, B, kappa, int(has_perm_q), int(has_perm_k)))


def _workspace(nbytes, device):
    torch = _torch()
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def ba_select_into(q, k, block, kappa, beta, sort_mode, sort_window, perm_q, perm_k, block_idx,
                   block_mask, block_scores, workspace):
    """ba_select writing caller-allocated tensors (no allocation)."""
    lib = load()
    _need_cuda(q, k, perm_q, perm_k, block_idx, block_mask, block_scores, workspace)
    b, h, L, d = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        st = lib.ba_select(_ptr(q), _ptr(k), b, h, L, d, block, kappa, float(beta), sort_mode, sort_window,
                           _ptr(perm_q), _ptr(perm_k), _ptr(block_idx), _ptr(block_mask),
                           _ptr(block_scores), _ptr(workspace), ws_bytes, _stream(q.device))
    _check(st, "ba_select")


def ba_select_isolated_into(q, k, block, prefill_len, kappa_prefill, kappa_generation, beta, sort_mode,
                            sort_window, perm_q, perm_k, block_idx, block_mask, block_scores, workspace):
    """ba_select_isolated writing caller-allocated tensors (no allocation)."""
    lib = load()
    _need_cuda(q, k, perm_q, perm_k, block_idx, block_mask, block_scores, workspace)
    b, h, L, d = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        st = lib.ba_select_isolated(_ptr(q), _ptr(k), b, h, L, d, block, prefill_len, kappa_prefill,
                                    kappa_generation, float(beta), sort_mode, sort_window, _ptr(perm_q),
                                    _ptr(perm_k), _ptr(block_idx), _ptr(block_mask), _ptr(block_scores),
                                    _ptr(workspace), ws_bytes, _stream(q.device))
    _check(st, "ba_select_isolated")


def ba_select_isolated(q, k, block, prefill_len, kappa_prefill, kappa_generation, beta=1.0,
                       sort_mode=SORT_QK, sort_window=0, return_scores=False, workspace=None):
    """Isolated selection (SparseD §3.3 Eq. 5-6 over BA-Att's block scores):
    per query block, kappa_prefill key blocks from [0, prefill_len) and
    kappa_generation from [prefill_len, L).  Returns the same dict as
    ba_select, block_idx holding kappa_prefill + kappa_generation ids."""
    torch = _torch()
    _need_cuda(q, k)
    b, h, L, d = q.shape
    N = -(-L // block)
    kappa = kappa_prefill + kappa_generation
    dev = q.device
    out = dict(
        perm_q=torch.empty((b, h, L), dtype=torch.int32, device=dev),
        perm_k=torch.empty((b, h, L), dtype=torch.int32, device=dev),
        block_idx=torch.empty((b, h, N, kappa), dtype=torch.int32, device=dev),
        block_mask=torch.empty((b, h, N, -(-N // 32)), dtype=torch.int32, device=dev),
        block_scores=torch.empty((b, h, N, N), dtype=torch.float32, device=dev) if return_scores else None,
    )
    if workspace is None:
        workspace = _workspace(select_workspace_size(b, h, L, d, block, kappa, sort_mode, sort_window), dev)
    ba_select_isolated_into(q, k, block, prefill_len, kappa_prefill, kappa_generation, beta, sort_mode,
                            sort_window, out["perm_q"], out["perm_k"], out["block_idx"], out["block_mask"],
                            out["block_scores"], workspace)
    if not return_scores:
        del out["block_scores"]
    return out


def ba_block_fidelity(q, k, block, lse, perm_q=None, perm_k=None, block_idx=None, scale=0.0,
                      deviation=True, bound=True):
    """Fidelity diagnostics of a selection (BA-Att §3.1 Eq. 3, §3.2 Eq. 5-8)
    over the sorted blocks of perm_q / perm_k (None = identity).  ``lse`` is
    the dense row LSE from ba_attn_dense.  Returns a dict with mass (fp32
    [b,h,N,N], Eq. 3), and as asked dev_max and bound ([b,h,N,N]) and recall
    ([b,h,N], when ``block_idx`` is given)."""
    torch = _torch()
    lib = load()
    _need_cuda(q, k, lse, perm_q, perm_k, block_idx)
    b, h, L, d = q.shape
    N = -(-L // block)
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(mass=torch.empty((b, h, N, N), **f32),
               dev_max=torch.empty((b, h, N, N), **f32) if deviation else None,
               bound=torch.empty((b, h, N, N), **f32) if bound else None,
               recall=torch.empty((b, h, N), **f32) if block_idx is not None else None)
    kappa = 0 if block_idx is None else block_idx.shape[-1]
    ws = _workspace(int(lib.ba_block_fidelity_workspace_size(b, h, L, d, block)), dev)
    ws_bytes = ws.numel() * ws.element_size()
    with _on_device(q):
        st = lib.ba_block_fidelity(_ptr(q), _ptr(k), b, h, L, d, block, _ptr(perm_q), _ptr(perm_k), _ptr(lse),
                                   float(scale), _ptr(block_idx), kappa, _ptr(out["mass"]), _ptr(out["dev_max"]),
                                   _ptr(out["bound"]), _ptr(out["recall"]), _ptr(ws), ws_bytes, _stream(dev))
    _check(st, "ba_block_fidelity")
    return {kk: vv for kk, vv in out.items() if vv is not None}


def ba_active_tokens(q_now, q_prev, group, top_k, return_mse=False):
    """LoSA locality pruning: uint8 [b,h,L] mask of the top_k tokens per
    group of ``group`` whose queries moved most between two steps (and the
    fp32 per-token MSE with ``return_mse``)."""
    torch = _torch()
    lib = load()
    _need_cuda(q_now, q_prev)
    b, h, L, d = q_now.shape
    active = torch.empty((b, h, L), dtype=torch.uint8, device=q_now.device)
    mse = torch.empty((b, h, L), dtype=torch.float32, device=q_now.device) if return_mse else None
    with _on_device(q_now):
        st = lib.ba_active_tokens(_ptr(q_now), _ptr(q_prev), b, h, L, d, group, top_k, _ptr(active),
                                  _ptr(mse), _stream(q_now.device))
    _check(st, "ba_active_tokens")
    return (active, mse) if return_mse else active


def ba_reuse_rows(o_new, lse_new, active, o_cache, lse_cache):
    """LoSA cache update in place: active rows of o_cache / lse_cache take
    o_new / lse_new."""
    lib = load()
    _need_cuda(o_new, lse_new, active, o_cache, lse_cache)
    d = o_new.shape[-1]
    rows = o_new.numel() // d
    with _on_device(o_new):
        st = lib.ba_reuse_rows(_ptr(o_new), _ptr(lse_new), _ptr(active), rows, d, _ptr(o_cache),
                               _ptr(lse_cache), _stream(o_new.device))
    _check(st, "ba_reuse_rows")


def ba_select_noalloc_into(q, k, block, kappa, beta, sort_mode, sort_window, perm_q, perm_k,
                           block_idx, block_mask, block_scores):
    """ba_select through the library's built-in scratch array (for callers that
    cannot allocate device memory); writes caller-allocated outputs."""
    lib = load()
    _need_cuda(q, k, perm_q, perm_k, block_idx, block_mask, block_scores)
    b, h, L, d = q.shape
    with _on_device(q):
        st = lib.ba_select_noalloc(_ptr(q), _ptr(k), b, h, L, d, block, kappa, float(beta), sort_mode,
                                   sort_window, _ptr(perm_q), _ptr(perm_k), _ptr(block_idx),
                                   _ptr(block_mask), _ptr(block_scores), _stream(q.device))
    _check(st, "ba_select_noalloc")


def ba_select(q, k, block, kappa, beta=1.0, sort_mode=SORT_QK, sort_window=0, return_scores=False,
              workspace=None):
    """Selection stage (BA-Att Algorithm 1 steps 1-11) on bf16 [b,h,L,d] q, k.

    Returns a dict with perm_q, perm_k (int32 [b,h,L]), block_idx (int32
    [b,h,N,kappa]), block_mask (int32 view of uint32 words [b,h,N,ceil(N/32)])
    and, with ``return_scores``, block_scores (fp32 [b,h,N,N]).
    """
    torch = _torch()
    _need_cuda(q, k)
    b, h, L, d = q.shape
    N = -(-L // block)
    dev = q.device
    out = dict(
        perm_q=torch.empty((b, h, L), dtype=torch.int32, device=dev),
        perm_k=torch.empty((b, h, L), dtype=torch.int32, device=dev),
        block_idx=torch.empty((b, h, N, kappa), dtype=torch.int32, device=dev),
        block_mask=torch.empty((b, h, N, -(-N // 32)), dtype=torch.int32, device=dev),
        block_scores=torch.empty((b, h, N, N), dtype=torch.float32, device=dev) if return_scores else None,
    )
    if workspace is None:
        workspace = _workspace(select_workspace_size(b, h, L, d, block, kappa, sort_mode, sort_window), dev)
    ba_select_into(q, k, block, kappa, beta, sort_mode, sort_window, out["perm_q"], out["perm_k"],
                   out["block_idx"], out["block_mask"], out["block_scores"], workspace)
    if not return_scores:
        del out["block_scores"]
    return out


def ba_sparse_attn_into(q, k, v, block, perm_q, perm_k, block_idx, scale, o, lse, workspace):
    lib = load()
    _need_cuda(q, k, v, perm_q, perm_k, block_idx, o, lse, workspace)
    b, h, L, d = q.shape
    kappa = block_idx.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        st = lib.ba_sparse_attn(_ptr(q), _ptr(k), _ptr(v), b, h, L, d, block, _ptr(perm_q), _ptr(perm_k),
                                _ptr(block_idx), kappa, float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
                                ws_bytes, _stream(q.device))
    _check(st, "ba_sparse_attn")


def ba_sparse_attn(q, k, v, block, perm_q, perm_k, block_idx, scale=0.0, workspace=None):
    """Block-sparse attention (Algorithm 1 step 12): returns (o bf16 [b,h,L,d], lse fp32 [b,h,L])."""
    torch = _torch()
    _need_cuda(q, k, v)
    b, h, L, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, L), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(sparse_attn_workspace_size(b, h, L, d, block, block_idx.shape[-1],
                                                          perm_q is not None, perm_k is not None), q.device)
    ba_sparse_attn_into(q, k, v, block, perm_q, perm_k, block_idx, scale, o, lse, workspace)
    return o, lse


def ba_attn_dense_into(q, k, v, scale, o, lse):
    lib = load()
    _need_cuda(q, k, v, o, lse)
    b, h, L, d = q.shape
    with _on_device(q):
        st = lib.ba_attn_dense(_ptr(q), _ptr(k), _ptr(v), b, h, L, d, float(scale), _ptr(o), _ptr(lse),
                               _stream(q.device))
    _check(st, "ba_attn_dense")


def ba_attn_dense(q, k, v, scale=0.0):
    """Dense attention with the same kernel: returns (o, lse)."""
    torch = _torch()
    _need_cuda(q, k, v)
    b, h, L, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, L), dtype=torch.float32, device=q.device)
    ba_attn_dense_into(q, k, v, scale, o, lse)
    return o, lse


def ba_merge_lse_into(o1, lse1, o2, lse2, o, lse):
    """Merge two results over disjoint key sets (LoSA merge); writes o, lse."""
    lib = load()
    _need_cuda(o1, lse1, o2, lse2, o, lse)
    d = o1.shape[-1]
    rows = o1.numel() // d
    with _on_device(o1):
        st = lib.ba_merge_lse(_ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), rows, d, _ptr(o), _ptr(lse),
                              _stream(o1.device))
    _check(st, "ba_merge_lse")


def ba_merge_lse(o1, lse1, o2, lse2):
    """Returns (o, lse) of the merged result; o1/o2 bf16 [..., d], lse fp32 [...]."""
    torch = _torch()
    o = torch.empty_like(o1)
    lse = torch.empty_like(lse1)
    ba_merge_lse_into(o1, lse1, o2, lse2, o, lse)
    return o, lse


def ba_validate_selection(block, block_idx, perm_q=None, perm_k=None):
    """Checks a selection on the device (pi_q, pi_k permutations; each row of
    block_idx strictly ascending with ids < N).  Returns (status, detail):
    status 0 when every check passes, else BA_ERR_INVALID_ARG (1) with detail
    bits 1 pi_q, 2 pi_k, 4 block_idx.  Synchronous."""
    lib = load()
    _need_cuda(block_idx, perm_q, perm_k)
    b, h, N, kappa = block_idx.shape
    L = perm_q.shape[-1] if perm_q is not None else (perm_k.shape[-1] if perm_k is not None else N * block)
    word = ctypes.c_uint32(0)
    with _on_device(block_idx):
        st = lib.ba_validate_selection(_ptr(perm_q), _ptr(perm_k), _ptr(block_idx), b, h, L, block, kappa,
                                       ctypes.byref(word), _stream(block_idx.device))
    if st not in (0, 1):
        raise BAError(st, "ba_validate_selection")
    return st, word.value


def selftest_wait_timeout(limit_us=1000, device=None):
    """Launch the bounded-wait self-test (a wait that runs out after
    ``limit_us``; no fault); read the result with last_device_error()."""
    torch = _torch()
    lib = load()
    _check(lib.ba_selftest_wait_timeout(int(limit_us), _stream(device or torch.device("cuda"))),
           "ba_selftest_wait_timeout")


def selftest_attn_stall(q, k, v, o, lse, limit_us=1000):
    """Run the dense attention kernel with its second K/V stage never loaded,
    so that the MMA thread's bounded wait runs out after ``limit_us`` and the
    kernel unwinds (no fault, nothing written to o / lse); read the result
    with last_device_error()."""
    lib = load()
    _need_cuda(q, k, v, o, lse)
    b, h, L, d = q.shape
    with _on_device(q):
        st = lib.ba_selftest_attn_stall(_ptr(q), _ptr(k), _ptr(v), b, h, L, d, int(limit_us), _ptr(o),
                                        _ptr(lse), _stream(q.device))
    _check(st, "ba_selftest_attn_stall")


def last_device_error(device=None):
    """Synchronise the current stream and return (status, raw error word)."""
    torch = _torch()
    lib = load()
    word = ctypes.c_uint32(0)
    st = lib.ba_last_device_error(_stream(device or torch.device("cuda")), ctypes.byref(word))
    return st, word.value
