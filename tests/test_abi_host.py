"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/ba.h declares, and rejects bad
arguments with the documented status before touching the device."""

import ctypes

import pytest

import block_sparse_bidirectional_gb300 as bsb

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3

# Plausible-looking device addresses: 256-byte aligned, never dereferenced
# because every call below fails its host checks first.
P = ctypes.c_void_p(0x10000000)
P2 = ctypes.c_void_p(0x20000000)
MIS = ctypes.c_void_p(0x10000004)  # not 16-byte aligned


def test_header_declares_the_documented_calls():
    names = set(bsb.header_functions())
    for n in ("ba_select", "ba_sparse_attn", "ba_attn_dense", "ba_select_workspace_size",
              "ba_sparse_attn_workspace_size", "ba_status_string", "ba_version",
              "ba_last_device_error"):
        assert n in names


def test_library_exports_every_header_function():
    lib = bsb.load()
    for name in bsb.header_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version():
    lib = bsb.load()
    assert lib.ba_status_string(0) == b"BA_OK"
    for s in range(1, 6):
        assert lib.ba_status_string(s).startswith(b"BA_ERR_")
    assert lib.ba_status_string(99) == b"BA_ERR_UNKNOWN"
    assert b"sm_103a" in lib.ba_version()


def test_workspace_sizes():
    lib = bsb.load()
    # no sort: no key buffers; stats (a, b) + scores scratch
    b, h, L, d, B = 1, 32, 65536, 128, 128
    N = L // B
    aug = b * h * N * 3 * d * 4
    sc = b * h * N * N * 4
    keys = 2 * b * h * L * 8
    assert lib.ba_select_workspace_size(b, h, L, d, B, 256, 0, 0) == 2 * aug + sc
    assert lib.ba_select_workspace_size(b, h, L, d, B, 256, 3, 0) == 2 * keys + 2 * aug + sc
    t = b * h * L * d * 2

    def a256(x):
        return (x + 255) // 256 * 256
    # tile-pair lists (uint16, two tiles of N entries per CTA) and their counts
    npairs = ((L + 127) // 128 + 1) // 2
    pl = a256(b * h * npairs * 2 * N * 2) + a256(b * h * npairs * 4 * 4)
    # with a permutation: the permuted copies and two gather counters per head
    rc = a256(b * h * 2 * 4)
    assert lib.ba_sparse_attn_workspace_size(b, h, L, d, B, 256, 1, 1) == 3 * t + pl + rc
    assert lib.ba_sparse_attn_workspace_size(b, h, L, d, B, 256, 0, 1) == 2 * t + pl + rc
    assert lib.ba_sparse_attn_workspace_size(b, h, L, d, B, 256, 0, 0) == pl
    # unsupported shapes report 0
    assert lib.ba_select_workspace_size(1, 1, 1024, 96, 64, 8, 3, 0) == 0
    assert lib.ba_select_workspace_size(1, 1, 1024, 64, 32, 8, 3, 0) == 0


def _select(lib, **kw):
    a = dict(q=P, k=P, b=1, h=1, L=1024, d=64, B=64, kappa=8, beta=1.0, mode=3, win=0,
             pq=P2, pk=P2, idx=P2, mask=P2, scores=None, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ba_select(a["q"], a["k"], a["b"], a["h"], a["L"], a["d"], a["B"], a["kappa"],
                         a["beta"], a["mode"], a["win"], a["pq"], a["pk"], a["idx"], a["mask"],
                         a["scores"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID),
    (dict(k=MIS), INVALID),
    (dict(idx=None), INVALID),
    (dict(mask=MIS), INVALID),
    (dict(kappa=0), INVALID),
    (dict(kappa=17), INVALID),
    (dict(mode=4), INVALID),
    (dict(win=100), INVALID),
    (dict(beta=float("nan")), INVALID),
    (dict(L=0), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(B=32), UNSUPPORTED),
    (dict(L=64 * 4097, kappa=8), UNSUPPORTED),
    (dict(ws_bytes=1024), WORKSPACE),
    (dict(ws=None), WORKSPACE),
    (dict(ws=ctypes.c_void_p(0x10000010)), WORKSPACE),
])
def test_select_rejects(kw, status):
    assert _select(bsb.load(), **kw) == status


def _select_iso(lib, **kw):
    a = dict(q=P, k=P, b=1, h=1, L=1024, d=64, B=64, pre=256, kpre=2, kgen=6, beta=1.0, mode=3,
             win=0, pq=P2, pk=P2, idx=P2, mask=P2, scores=None, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ba_select_isolated(a["q"], a["k"], a["b"], a["h"], a["L"], a["d"], a["B"], a["pre"],
                                  a["kpre"], a["kgen"], a["beta"], a["mode"], a["win"], a["pq"],
                                  a["pk"], a["idx"], a["mask"], a["scores"], a["ws"], a["ws_bytes"],
                                  a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(pre=0), INVALID),             # no prefill part
    (dict(pre=1024), INVALID),          # no generation part
    (dict(pre=100), INVALID),           # not a multiple of the block
    (dict(kpre=0), INVALID),
    (dict(kpre=5), INVALID),            # more than the 4 prefill blocks
    (dict(kgen=0), INVALID),
    (dict(kgen=13), INVALID),           # more than the 12 generation blocks
    (dict(q=None), INVALID),
    (dict(mask=MIS), INVALID),
    (dict(mode=4), INVALID),
    (dict(win=100), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(ws_bytes=1024), WORKSPACE),
])
def test_select_isolated_rejects(kw, status):
    assert _select_iso(bsb.load(), **kw) == status


def _fid(lib, **kw):
    a = dict(q=P, k=P, b=1, h=1, L=1024, d=64, B=64, pq=P2, pk=P2, lse=P, scale=0.0, idx=P2, kappa=8,
             mass=P, dev=P, bound=P, recall=P, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ba_block_fidelity(a["q"], a["k"], a["b"], a["h"], a["L"], a["d"], a["B"], a["pq"], a["pk"],
                                 a["lse"], a["scale"], a["idx"], a["kappa"], a["mass"], a["dev"],
                                 a["bound"], a["recall"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(lse=None), INVALID),
    (dict(mass=None), INVALID),
    (dict(q=None), INVALID),
    (dict(idx=None), INVALID),          # recall asked for without a list
    (dict(kappa=0), INVALID),
    (dict(kappa=17), INVALID),
    (dict(dev=MIS), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(d=96), UNSUPPORTED),
    (dict(B=32), UNSUPPORTED),
    (dict(ws_bytes=1024), WORKSPACE),
    (dict(ws=None), WORKSPACE),
])
def test_fidelity_rejects(kw, status):
    assert _fid(bsb.load(), **kw) == status


def test_fidelity_workspace_size():
    lib = bsb.load()
    b, h, L, d, B = 1, 4, 1000, 128, 64
    N = -(-L // B)

    def a256(x):
        return (x + 255) // 256 * 256
    want = (2 * a256(b * h * L * d * 2) + 2 * a256(b * h * N * d * 4) + 4 * a256(b * h * N * 4)
            + a256(b * h * N * N * 4))
    assert lib.ba_block_fidelity_workspace_size(b, h, L, d, B) == want
    assert lib.ba_block_fidelity_workspace_size(b, h, L, 96, B) == 0


def _act(lib, **kw):
    a = dict(qn=P, qp=P, b=1, h=2, L=1000, d=128, group=32, k=4, act=P2, mse=None, stream=None)
    a.update(kw)
    return lib.ba_active_tokens(a["qn"], a["qp"], a["b"], a["h"], a["L"], a["d"], a["group"], a["k"],
                                a["act"], a["mse"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(qn=None), INVALID),
    (dict(qp=MIS), INVALID),
    (dict(act=None), INVALID),
    (dict(group=0), INVALID),
    (dict(group=1025), INVALID),
    (dict(k=0), INVALID),
    (dict(L=0), INVALID),
    (dict(d=96), UNSUPPORTED),
])
def test_active_tokens_rejects(kw, status):
    assert _act(bsb.load(), **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(o_new=None), INVALID),
    (dict(o_cache=MIS), INVALID),
    (dict(act=None), INVALID),
    (dict(rows=-1), INVALID),
    (dict(d=32), UNSUPPORTED),
])
def test_reuse_rows_rejects(kw, status):
    a = dict(o_new=P, lse_new=P, act=P2, rows=100, d=64, o_cache=P, lse_cache=P, stream=None)
    a.update(kw)
    assert bsb.load().ba_reuse_rows(a["o_new"], a["lse_new"], a["act"], a["rows"], a["d"],
                                    a["o_cache"], a["lse_cache"], a["stream"]) == status


def _attn(lib, **kw):
    a = dict(q=P, k=P, v=P, b=1, h=1, L=1024, d=64, B=64, pq=P2, pk=P2, idx=P2, kappa=8, scale=0.0,
             o=P, lse=P, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ba_sparse_attn(a["q"], a["k"], a["v"], a["b"], a["h"], a["L"], a["d"], a["B"],
                              a["pq"], a["pk"], a["idx"], a["kappa"], a["scale"], a["o"], a["lse"],
                              a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(v=None), INVALID),
    (dict(o=MIS), INVALID),
    (dict(pq=MIS), INVALID),
    (dict(kappa=0), INVALID),
    (dict(kappa=17), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(d=80), UNSUPPORTED),
    (dict(B=256), UNSUPPORTED),
    (dict(ws_bytes=16), WORKSPACE),
])
def test_sparse_attn_rejects(kw, status):
    assert _attn(bsb.load(), **kw) == status


def test_dense_rejects():
    lib = bsb.load()
    assert lib.ba_attn_dense(None, P, P, 1, 1, 128, 64, 0.0, P, P, None) == INVALID
    assert lib.ba_attn_dense(P, P, P, 1, 1, 128, 72, 0.0, P, P, None) == UNSUPPORTED
    assert lib.ba_attn_dense(P, P, P, 1, 1, 0, 64, 0.0, P, P, None) == INVALID
    assert lib.ba_attn_dense(P, P, P, 1, 1, 128, 64, 0.0, MIS, P, None) == INVALID


def test_no_cpu_path():
    """The binding refuses CPU tensors instead of computing anything on the host."""
    import torch
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        bsb.ba_attn_dense(q, q, q)
    with pytest.raises(ValueError):
        bsb.ba_select(q, q, 64, 1)


def test_merge_lse_rejects():
    lib = bsb.load()
    assert lib.ba_merge_lse(P, P, P, P, 0, 128, P, P, None) == OK          # no rows: no-op
    assert lib.ba_merge_lse(P, P, P, P, -1, 128, P, P, None) == INVALID
    assert lib.ba_merge_lse(P, P, P, P, 10, 96, P, P, None) == UNSUPPORTED
    assert lib.ba_merge_lse(None, P, P, P, 10, 128, P, P, None) == INVALID
    assert lib.ba_merge_lse(P, P, MIS, P, 10, 64, P, P, None) == INVALID


def test_selftest_rejects_limits_outside_range():
    lib = bsb.load()
    for bad in (0, 1000001, 2**32 - 1):
        assert lib.ba_selftest_wait_timeout(bad, None) == INVALID


def test_validate_selection_rejects_before_launch():
    lib = bsb.load()
    u = ctypes.c_uint32(7)
    # block_idx is required; kappa within [1, N]; block 64 or 128; aligned pointers
    assert lib.ba_validate_selection(P, P, None, 1, 1, 1024, 64, 8, ctypes.byref(u), None) == INVALID
    assert u.value == 0
    assert lib.ba_validate_selection(P, P, P, 1, 1, 1024, 64, 0, None, None) == INVALID
    assert lib.ba_validate_selection(P, P, P, 1, 1, 1024, 64, 17, None, None) == INVALID
    assert lib.ba_validate_selection(P, P, P, 1, 1, 1024, 32, 8, None, None) == UNSUPPORTED
    assert lib.ba_validate_selection(MIS, P, P, 1, 1, 1024, 64, 8, None, None) == INVALID
    assert lib.ba_validate_selection(P, P, MIS, 1, 1, 1024, 64, 8, None, None) == INVALID
