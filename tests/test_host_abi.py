"""Host-side tests of the C ABI (no GPU): the library builds and loads, exports
every function include/muon.h declares, the ctypes structs match the C
layout, grouping matches the oracle's statement, and host-detectable argument
errors return before anything is enqueued."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import newton_schulz_02_gb300 as m
import oracle
from newton_schulz_02_gb300 import build as nbuild
from tests.conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "muon.h")


@pytest.fixture(scope="module")
def lib():
    nbuild.build()
    return m.load_library()


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["muon_step_batched", "newton_schulz_batched", "muon_group_by_shape",
              "muon_step_workspace_size", "newton_schulz_workspace_size", "muon_get_status",
              "muon_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing
    assert set(declared_functions()) <= set(m.PROTOTYPES)


def test_struct_layouts_match_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "muon.h"\n'
        "#define P(T) printf(#T \" %zu\\n\", sizeof(T));\n"
        "#define O(T,f) printf(#T \".\" #f \" %zu\\n\", offsetof(T,f));\n"
        "int main(void){P(muon_ns_stage_t)P(muon_ns_schedule_t)P(muon_view_t)P(muon_group_t)"
        "P(muon_hparams_t)P(muon_tensor_desc_t)P(muon_adamw_group_t)P(muon_adamw_hparams_t)"
        "O(muon_adamw_group_t,numel)O(muon_adamw_group_t,w_ptrs)O(muon_adamw_group_t,wd_mask)"
        "O(muon_adamw_hparams_t,weight_decay)O(muon_adamw_hparams_t,t)"
        "O(muon_group_t,view)O(muon_group_t,w_ptrs)O(muon_group_t,wd_mask)"
        "O(muon_hparams_t,t)O(muon_hparams_t,lr)O(muon_view_t,row_stride)"
        "O(muon_view_t,fan_out_axis)O(muon_tensor_desc_t,w_dtype)"
        "O(muon_ns_schedule_t,prec)O(muon_ns_schedule_t,merge_groups)return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(prog),
                           "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    for name in ["muon_ns_stage_t", "muon_ns_schedule_t", "muon_view_t", "muon_group_t",
                 "muon_hparams_t", "muon_tensor_desc_t", "muon_adamw_group_t",
                 "muon_adamw_hparams_t"]:
        assert int(got[name]) == ctypes.sizeof(getattr(m, name)), name
    for key, val in got.items():
        if "." in key:
            t, f = key.split(".")
            assert getattr(getattr(m, t), f).offset == int(val), key


def test_status_strings(lib):
    assert m.status_string(m.MUON_OK) == "MUON_OK"
    assert m.status_string(m.MUON_ERR_TIMEOUT) == "MUON_ERR_TIMEOUT"
    assert m.status_string(99) == "MUON_ERR_UNKNOWN"


def test_hybrid_schedule_matches_page(lib):
    s = m.muon_ns_hybrid_schedule()
    got = tuple((s.stages[i].steps, (s.stages[i].a, s.stages[i].b, s.stages[i].c))
                for i in range(s.n_stages))
    want = tuple((int(r[0]), tuple(float(np.float32(v)) for v in r[1:]))
                 for r in read_golden("hybrid_schedule.txt"))
    assert got == want and s.normalize == 1 and s.prec == m.MUON_NS_BF16


def test_group_by_shape_matches_golden_and_oracle(lib):
    K0, K1, K2 = (1024, 1024, 1024, 0, 0, 0), (1024, 4096, 4096, 0, 0, 0), (8, 16, 16, 0, 0, 0)
    keys = [K0, K1, K0, K0, K2, K1]
    for row in read_golden("group_by_shape.txt"):
        mb, ng = int(row[0]), int(row[1])
        got, n = m.muon_group_by_shape(keys, mb)
        assert (got, n) == ([int(v) for v in row[2:]], ng)
    rng = np.random.default_rng(0)
    pool = [(r, c, c, wd, gd, ax) for r in (8, 16) for c in (8, 24) for wd in (0, 1)
            for gd in (0, 1) for ax in (0, 1)]
    for trial in range(50):
        n = int(rng.integers(0, 40))
        keys = [pool[int(i)] for i in rng.integers(0, len(pool), size=n)]
        mb = int(rng.integers(0, 5))
        assert m.muon_group_by_shape(keys, mb) == oracle.group_by_shape(keys, mb)


def test_group_by_shape_errors(lib):
    L = m.load_library()
    ng = ctypes.c_int()
    assert L.muon_group_by_shape(None, 1, 0, None, ctypes.byref(ng)) == m.MUON_ERR_INVALID_ARG
    assert L.muon_group_by_shape(None, 0, -1, None, ctypes.byref(ng)) == m.MUON_ERR_INVALID_ARG
    assert L.muon_group_by_shape(None, 0, 0, None, ctypes.byref(ng)) == m.MUON_OK and ng.value == 0


def _group(rows, cols, row_stride=None, batch=1, wdt=0, gdt=0, ptr=0x1000):
    g = m.muon_group_t()
    g.batch = batch
    g.view = m.muon_view_t(rows, cols, cols if row_stride is None else row_stride, 0, 0)
    g.w_dtype, g.g_dtype = wdt, gdt
    g.w_ptrs = g.g_ptrs = g.m_ptrs = ptr
    g.wd_mask = None
    return g


def _ws_size(groups, sched=None):
    arr = (m.muon_group_t * len(groups))(*groups)
    nb = ctypes.c_size_t()
    code = m.load_library().muon_step_workspace_size(arr, len(groups), sched, ctypes.byref(nb))
    return code, nb.value


def test_workspace_size_layout(lib):
    code, nb = _ws_size([_group(1024, 1024, batch=64)])
    assert code == m.MUON_OK
    x = 64 * 1024 * 1024 * 2
    assert 6 * x < nb < 6 * x + (1 << 20)      # X ping-pong (hi + lo planes) + S + P + vectors
    code2, nb2 = _ws_size([_group(1024, 1024, batch=64), _group(100, 64, batch=3)])
    assert code2 == m.MUON_OK and nb2 == nb     # groups reuse the workspace: max, not sum
    code3, nb3 = _ws_size([_group(4096, 128, row_stride=4096, batch=32)])
    assert code3 == m.MUON_OK
    assert nb3 > 4 * 32 * 128 * 4096 * 2        # tall heads run as wide 128 x 4096


@pytest.mark.parametrize("rows,cols,rs,want", [
    (0, 8, 8, m.MUON_ERR_INVALID_ARG),
    (8, 8, 4, m.MUON_ERR_INVALID_ARG),
    (8, 12, 12, m.MUON_ERR_UNSUPPORTED),
    (8, 8, 12, m.MUON_ERR_MISALIGNED),
    (3, 8, 8, m.MUON_OK),
    (1 << 20, 8, 8, m.MUON_OK),                       # the largest side the library takes
    (8, 1 << 20, 1 << 20, m.MUON_OK),
    ((1 << 20) + 8, 8, 8, m.MUON_ERR_INVALID_ARG),    # beyond it: rejected, not truncated
    (8, (1 << 20) + 8, (1 << 20) + 8, m.MUON_ERR_INVALID_ARG),
])
def test_view_validation(lib, rows, cols, rs, want):
    code, _ = _ws_size([_group(rows, cols, rs)])
    assert code == want


def test_merged_chains_workspace(lib):
    """merge_groups: a 1024 x 4096 group and a 4096 x 1024 group share one
    chain, so the workspace holds both batches at once; unmerged it holds the
    larger group only.  Groups of another wide shape stay apart."""
    merged = m.Schedule(oracle_hybrid(), merge_groups=True)
    plain = m.Schedule(oracle_hybrid())
    gs = [_group(1024, 4096, batch=8), _group(4096, 1024, batch=8), _group(512, 512, batch=2)]
    c0, nb0 = _ws_size(gs, plain.ref)
    c1, nb1 = _ws_size(gs, merged.ref)
    one = _ws_size([_group(1024, 4096, batch=16)], plain.ref)[1]
    assert c0 == c1 == m.MUON_OK
    assert nb0 == _ws_size([_group(1024, 4096, batch=8)], plain.ref)[1]
    assert nb1 == one
    five = [_group(1024, 4096, batch=1) for _ in range(5)]      # chains of at most 4 groups
    assert _ws_size(five, merged.ref)[1] == _ws_size([_group(1024, 4096, batch=4)], plain.ref)[1]
    bad = m.Schedule(oracle_hybrid())
    bad.c.merge_groups = 2
    assert _ws_size(gs, bad.ref)[0] == m.MUON_ERR_INVALID_ARG


def oracle_hybrid():
    return [(8, (3.4445, -4.7750, 2.0315)), (2, (2.0, -1.5, 0.5))]


def test_split_bf16_workspace_adds_lo_planes_of_s_and_p(lib):
    """The split-bf16 layout adds lo planes of S and P, and drops the ticket
    counters and log of the fused bf16 Gram + polynomial launches (64
    counters, then 128 rows of one launch's tickets + 2: 2 x 64 matrices x
    10 upper 256 x 256 super-blocks of a 1024^2 Gram)."""
    x3 = m.Schedule([(1, (1.0, 0.0, 0.0))], prec=m.MUON_NS_BF16X3)
    code, nb = _ws_size([_group(1024, 1024, batch=64)])
    code3, nb3 = _ws_size([_group(1024, 1024, batch=64)], x3.ref)
    assert code == code3 == m.MUON_OK
    log_bytes = (64 + 128 * (2 * 64 * 10 + 2)) * 4
    assert nb3 == nb + 2 * 64 * 1024 * 1024 * 2 - (log_bytes + 255) // 256 * 256


def test_schedule_validation(lib):
    tf32 = m.Schedule([(1, (1.0, 0.0, 0.0))], prec=m.MUON_NS_TF32)
    assert _ws_size([_group(8, 8)], tf32.ref)[0] == m.MUON_ERR_UNSUPPORTED
    other = m.Schedule([(1, (1.0, 0.0, 0.0))], prec=7)
    assert _ws_size([_group(8, 8)], other.ref)[0] == m.MUON_ERR_INVALID_ARG
    bad = m.Schedule([(-1, (1.0, 0.0, 0.0))])
    assert _ws_size([_group(8, 8)], bad.ref)[0] == m.MUON_ERR_INVALID_ARG
    nan = m.Schedule([(1, (float("nan"), 0.0, 0.0))])
    assert _ws_size([_group(8, 8)], nan.ref)[0] == m.MUON_ERR_INVALID_ARG


def _step(groups, hp, ws_ptr, ws_bytes):
    arr = (m.muon_group_t * len(groups))(*groups)
    return m.load_library().muon_step_batched(arr, len(groups), ctypes.byref(hp), None, ws_ptr,
                                              ws_bytes, None)


def test_step_rejects_before_enqueue(lib):
    """Every case returns before the library touches CUDA (no GPU here)."""
    hp = m.hparams()
    g = _group(64, 64)
    _, need = _ws_size([g])
    assert _step([g], hp, 0x100000, need - 1) == m.MUON_ERR_WORKSPACE_TOO_SMALL
    assert _step([g], hp, 0x100010, need) == m.MUON_ERR_MISALIGNED
    assert _step([g], hp, None, need) == m.MUON_ERR_INVALID_ARG
    assert _step([_group(64, 64, ptr=0)], hp, 0x100000, need) == m.MUON_ERR_INVALID_ARG
    assert _step([_group(64, 64, wdt=7)], hp, 0x100000, need) == m.MUON_ERR_INVALID_ARG
    bad_hp = m.hparams(lr=float("inf"))
    assert _step([g], bad_hp, 0x100000, need) == m.MUON_ERR_INVALID_ARG
    ema0 = m.hparams(style="ema", t=0)
    assert _step([g], ema0, 0x100000, need) == m.MUON_ERR_INVALID_ARG
    L = m.load_library()
    assert L.muon_step_batched(None, 1, ctypes.byref(hp), None, 0x100000, need, None) == \
        m.MUON_ERR_INVALID_ARG
    # a group of no matrices is an error (an empty call passes no groups instead)
    assert _step([_group(64, 64, batch=0)], hp, 0x100000, need) == m.MUON_ERR_INVALID_ARG
    assert _ws_size([_group(64, 64, batch=0)])[0] == m.MUON_ERR_INVALID_ARG


def test_adamw_rejects_before_enqueue(lib):
    """Host-detectable AdamW errors return before any CUDA call (no GPU here)."""
    L = m.load_library()
    g = m.muon_adamw_group_t(2, 100, m.MUON_BF16, m.MUON_BF16, 0x1000, 0x2000, 0x3000, 0x4000, None)
    arr = (m.muon_adamw_group_t * 1)(g)
    call = lambda a, n, hp, flags=None: L.muon_adamw_step(a, n, ctypes.byref(hp), flags, None)
    hp = m.adamw_hparams()
    assert call(arr, 1, m.adamw_hparams(t=0)) == m.MUON_ERR_INVALID_ARG
    assert call(arr, 1, m.adamw_hparams(beta1=1.0)) == m.MUON_ERR_INVALID_ARG
    assert call(arr, 1, m.adamw_hparams(beta2=-0.1)) == m.MUON_ERR_INVALID_ARG
    assert call(arr, 1, m.adamw_hparams(eps=-1e-8)) == m.MUON_ERR_INVALID_ARG
    assert call(arr, 1, m.adamw_hparams(lr=float("nan"))) == m.MUON_ERR_INVALID_ARG
    assert call(arr, 1, hp, 0x1002) == m.MUON_ERR_MISALIGNED
    assert call(None, 1, hp) == m.MUON_ERR_INVALID_ARG
    assert call(arr, -1, hp) == m.MUON_ERR_INVALID_ARG
    for bad in (m.muon_adamw_group_t(-1, 100, 0, 0, 0x1000, 0x2000, 0x3000, 0x4000, None),
                m.muon_adamw_group_t(2, -5, 0, 0, 0x1000, 0x2000, 0x3000, 0x4000, None),
                m.muon_adamw_group_t(2, 100, 9, 0, 0x1000, 0x2000, 0x3000, 0x4000, None),
                m.muon_adamw_group_t(2, 100, 0, 0, 0x1000, None, 0x3000, 0x4000, None)):
        assert call((m.muon_adamw_group_t * 1)(bad), 1, hp) == m.MUON_ERR_INVALID_ARG
    # empty groups enqueue nothing
    empty = m.muon_adamw_group_t(0, 100, 0, 0, None, None, None, None, None)
    assert call((m.muon_adamw_group_t * 1)(empty), 1, hp) == m.MUON_OK
    assert call(arr, 0, hp) == m.MUON_OK


def test_newton_schulz_rejects_before_enqueue(lib):
    L = m.load_library()
    v = m.muon_view_t(64, 64, 64, 64 * 64, 0)
    nb = ctypes.c_size_t()
    assert L.newton_schulz_workspace_size(ctypes.byref(v), 2, None, ctypes.byref(nb)) == m.MUON_OK
    need = nb.value
    args = lambda x, o, ws, n: (x, m.MUON_BF16, ctypes.byref(v), 2, o, m.MUON_F32, None, ws, n, None)
    assert L.newton_schulz_batched(*args(0x200008, 0x900000, 0x100000, need)) == m.MUON_ERR_MISALIGNED
    assert L.newton_schulz_batched(*args(0x200000, 0x900000, 0x100000, need - 1)) == \
        m.MUON_ERR_WORKSPACE_TOO_SMALL
    assert L.newton_schulz_batched(*args(0x200000, 0x200000, 0x100000, need)) == \
        m.MUON_ERR_INVALID_ARG                   # x and out overlap
    assert L.newton_schulz_batched(*args(None, 0x900000, 0x100000, need)) == m.MUON_ERR_INVALID_ARG
    # batch 0 is rejected by the size query and by the call
    assert L.newton_schulz_workspace_size(ctypes.byref(v), 0, None, ctypes.byref(nb)) == \
        m.MUON_ERR_INVALID_ARG
    assert L.newton_schulz_batched(0x200000, m.MUON_BF16, ctypes.byref(v), 0, 0x900000, m.MUON_F32,
                                   None, 0x100000, need, None) == m.MUON_ERR_INVALID_ARG


def test_timeout_setting(lib):
    L = m.load_library()
    assert L.muon_set_wait_timeout_ns(0) == m.MUON_ERR_INVALID_ARG
    assert L.muon_set_wait_timeout_ns(2_000_000_000) == m.MUON_OK
    assert L.muon_check_wait_timeout(0x100000, 256, 0, None) == m.MUON_ERR_INVALID_ARG
    assert L.muon_check_wait_timeout(0x100008, 256, 1000, None) == m.MUON_ERR_MISALIGNED


def test_binding_fails_loudly_without_library(tmp_path):
    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            m.load_library(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_occupy_sms_rejects_out_of_range_arguments(lib):
    L = m.load_library()
    assert L.muon_occupy_sms(0, 1024, 1000, None) == m.MUON_ERR_INVALID_ARG
    assert L.muon_occupy_sms(4, 228 << 10, 1000, None) == m.MUON_ERR_INVALID_ARG
    assert L.muon_occupy_sms(4, 1024, 0, None) == m.MUON_ERR_INVALID_ARG
    assert L.muon_occupy_sms(4, 1024, 2_000_000_000, None) == m.MUON_ERR_INVALID_ARG
