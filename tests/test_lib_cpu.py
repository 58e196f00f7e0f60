"""The C-ABI library without a GPU: it loads, exports every symbol rq.h declares,
and its host-side checks answer before any device work.

Pointers passed below are never dereferenced: each call fails a host-side check
first (shape, alignment, capacity) or is a pure host computation."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rq():
    import __graft_entry__
    __graft_entry__.build()
    import decode_attention_rq_gb300
    return decode_attention_rq_gb300


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "rq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", src))


def test_exports_every_declared_symbol(rq):
    declared = _declared_symbols()
    assert declared == set(rq.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(rq.lib, name), name


def test_status_strings(rq):
    for s in range(8):
        assert rq.rq_status_string(s)
    assert rq.rq_status_string(99) == "unknown status"


def _cfg(rq, **kw):
    base = dict(num_layers=24, loops_per_group=4, num_groups=1, num_heads=16, head_dim=128,
                group_size=32, max_batch=4, max_seq_len=8192, mode=0)
    base.update(kw)
    return rq.rq_config(**base)


def test_cache_bytes_matches_storage_accounting(rq):
    import oracle
    cfg = _cfg(rq)
    n = rq.rq_cache_bytes(cfg)
    # 396 bytes per token per (layer, row, head) for d=128, g=32, 4 loops
    assert n == 24 * 4 * 16 * 8192 * 396
    geom = oracle.Geometry(24, 4, 1, 16, 128, 32, 4, 8192)
    assert n == geom.total_bytes
    for d, g, P, G, N in [(96, 32, 4, 8, 4096), (128, 16, 4, 1, 1000), (96, 16, 2, 3, 77), (128, 32, 1, 1, 64),
                          (96, 32, 8, 4, 4096), (96, 32, 16, 2, 4096), (128, 16, 16, 1, 300)]:
        cfg = _cfg(rq, head_dim=d, group_size=g, loops_per_group=P, num_groups=G, max_seq_len=N)
        assert rq.rq_cache_bytes(cfg) == oracle.Geometry(24, P, G, 16, d, g, 4, N).total_bytes


@pytest.mark.parametrize("kw", [dict(head_dim=64), dict(group_size=8), dict(head_dim=96, group_size=64),
                                dict(loops_per_group=0), dict(loops_per_group=17), dict(mode=8),
                                dict(head_dim=96, mode=4), dict(num_heads=0), dict(max_seq_len=0)])
def test_unsupported_shapes(rq, kw):
    cfg = _cfg(rq, **kw)
    assert rq.rq_cache_bytes(cfg) == 0
    h = ctypes.c_void_p()
    st = rq.lib.rq_cache_create(ctypes.byref(cfg), 0x1000, 1 << 40, 0x2000, ctypes.byref(h))
    assert st == 6  # RQ_ERR_UNSUPPORTED


def test_create_argument_checks(rq):
    cfg = _cfg(rq, num_layers=1, max_seq_len=64, max_batch=1, num_heads=1)
    need = rq.rq_cache_bytes(cfg)
    h = ctypes.c_void_p()
    assert rq.lib.rq_cache_create(ctypes.byref(cfg), None, need, 0x2000, ctypes.byref(h)) == 1
    assert rq.lib.rq_cache_create(ctypes.byref(cfg), 0x1000, need - 1, 0x2000, ctypes.byref(h)) == 3
    assert rq.lib.rq_cache_create(ctypes.byref(cfg), 0x1008, need, 0x2000, ctypes.byref(h)) == 2
    assert rq.lib.rq_cache_create(ctypes.byref(cfg), 0x1000, need, 0x2004, ctypes.byref(h)) == 2
    assert rq.lib.rq_cache_destroy(None) == 0
    # the rotation may be NULL only with the Walsh-Hadamard mode (which needs d = 128)
    assert rq.lib.rq_cache_create(ctypes.byref(cfg), 0x1000, need, None, ctypes.byref(h)) == 1
    hcfg = _cfg(rq, num_layers=1, max_seq_len=64, max_batch=1, num_heads=1, mode=rq.RQ_MODE_HADAMARD)
    assert rq.rq_cache_bytes(hcfg) == need


def test_bf16_argument_checks(rq):
    p = 0x10000
    f = rq.lib.rq_decode_attention_bf16
    assert f(p, p, p, p, p, p, 2, 4, 64, 100, 0.1, p, p, 1 << 30, None) == 6      # head_dim
    assert f(p, p, p, p, p, None, 2, 4, 128, 100, 0.1, p, p, 1 << 30, None) == 1  # null
    assert f(p, p, p, p, p, p, 0, 4, 128, 100, 0.1, p, p, 1 << 30, None) == 1     # batch
    assert f(p, p, p, p, p, p, 257, 4, 128, 100, 0.1, p, p, 1 << 30, None) == 6   # above RQ_MAX_DECODE_BATCH
    assert rq.rq_bf16_workspace_bytes(2, 4, 64) == 0


def test_decode_argument_checks_need_no_device(rq):
    f = rq.lib.rq_decode_attention
    p = 0x10000
    assert f(None, 0, 0, 0, 1, p, p, p, p, 0.1, p, p, 1 << 20, None) == 1
    assert rq.lib.rq_append(None, 0, 0, 1, p, p, 1, None, None) == 1
