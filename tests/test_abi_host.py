"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import exact_attention_blackwell_tiled_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P16 = ctypes.c_void_p(16 * 1024)  # aligned, never dereferenced: validation fails first
P17 = ctypes.c_void_p(16 * 1024 + 1)


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return fa.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert declared, "no declarations parsed"
    assert declared == set(fa.EXPORTS), declared ^ set(fa.EXPORTS)
    for name in declared:
        assert hasattr(L, name), f"libfa.so does not export {name}"


def test_status_strings(L):
    for code, name in fa.STATUS_NAMES.items():
        assert L.fa_status_string(code).decode() == name
    assert L.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


def _fwd(L, q=P16, k=P16, v=P16, o=P16, lse=P16, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, D=64, causal=0,
         scale=0.125):
    return L.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, None)


def test_fwd_rejects_bad_arguments(L):
    assert _fwd(L, q=None) == 1
    assert _fwd(L, lse=None) == 1
    assert _fwd(L, B=0) == 1
    assert _fwd(L, Hq=0) == 1
    assert _fwd(L, Sk=0) == 1
    assert _fwd(L, Sq=-1) == 1
    assert _fwd(L, Hq=3, Hkv=2) == 1
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, D=96) == 2
    assert _fwd(L, D=256) == 2
    assert _fwd(L, q=P17) == 3
    assert _fwd(L, o=P17) == 3
    # Sq == 0 is a no-op that needs no device
    assert _fwd(L, Sq=0) == 0
    assert L.fa_last_launch_count() == 0


def test_bwd_rejects_bad_arguments(L):
    need = L.fa_bwd_workspace_bytes(1, 2, 2, 8, 8, 64, 0)
    assert need > 0

    def call(ws=P16, ws_bytes=need, **kw):
        a = dict(q=P16, k=P16, v=P16, o=P16, do=P16, lse=P16, dq=P16, dk=P16, dv=P16, B=1, Hq=2,
                 Hkv=2, Sq=8, Sk=8, D=64, causal=0, scale=0.125, det=0)
        a.update(kw)
        return L.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                        a["dv"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["D"], a["causal"],
                        a["scale"], ws, ws_bytes, a["det"], None)

    assert call(dq=None) == 1
    assert call(Hq=4, Hkv=3) == 1
    assert call(D=80) == 2
    assert call(dk=P17) == 3
    assert call(ws=None) == 4
    assert call(ws_bytes=need - 1) == 4
    assert call(ws=ctypes.c_void_p(16 * 1024 + 16)) == 4  # workspace must be 256-byte aligned


def test_workspace_size(L):
    assert L.fa_bwd_workspace_bytes(0, 1, 1, 8, 8, 64, 0) == 0
    assert L.fa_bwd_workspace_bytes(1, 1, 1, 8, 8, 72, 0) == 0
    small = L.fa_bwd_workspace_bytes(1, 2, 2, 100, 100, 64, 0)
    big = L.fa_bwd_workspace_bytes(2, 16, 16, 8192, 8192, 128, 1)
    assert 0 < small < big
    # fp32 dQ accumulator dominates: B*Hq*Sq_pad*D*4
    assert big >= 2 * 16 * 8192 * 128 * 4
    assert big % 256 == 0


def test_row_count_limit(L):
    # rows over all heads are 32-bit in the kernels: B * Hq * ceil128(Sq) < 2^31
    assert L.fa_bwd_workspace_bytes(1 << 14, 1, 1, 1 << 17, 128, 64, 0) == 0
    assert L.fa_bwd_workspace_bytes(1, 1, 1, 128, 1 << 17, 64, 0) > 0
    assert L.fa_fwd(P16, P16, P16, P16, P16, 4, 1, 1, 128, 1 << 30, 64, 0, 1.0, None) == 1
    assert L.fa_fwd(P16, P16, P16, P16, P16, 1 << 13, 2, 1, 1 << 17, 128, 64, 0, 1.0, None) == 1


def test_score_mod_validation(L):
    bad = fa.ScoreMod(-1, 0, 16 * 1024 + 2)  # slopes must be 4-byte aligned
    assert L.fa_fwd_mod(P16, P16, P16, P16, P16, 1, 1, 1, 128, 128, 64, ctypes.byref(bad), 1.0,
                        None) == 3
    bad = fa.ScoreMod(-1, -1, None, 16 * 1024 + 1)  # key counts must be 4-byte aligned
    assert L.fa_fwd_mod(P16, P16, P16, P16, P16, 2, 1, 1, 128, 128, 64, ctypes.byref(bad), 1.0,
                        None) == 3
    assert L.fa_bwd_mod(P16, P16, P16, P16, P16, P16, P16, P16, P16, 2, 1, 1, 128, 128, 64,
                        ctypes.byref(bad), 1.0, P16, 1 << 30, 0, None) == 3
    # a window that leaves the last rows with no key is accepted (they get O = 0
    # and LSE = -inf); with Sq = 0 the call reads and writes nothing
    ok = fa.ScoreMod(64, -1, None, None)
    assert L.fa_fwd_mod(None, P16, P16, None, None, 1, 1, 1, 0, 128, 64, ctypes.byref(ok), 1.0,
                        None) == 0


def test_score_mod_layout():
    """The ctypes mirror of fa_score_mod matches the C layout: two ints, then the
    two device pointers."""
    assert ctypes.sizeof(fa.ScoreMod) == 24
    assert fa.ScoreMod.alibi_slopes.offset == 8 and fa.ScoreMod.seqlens_k.offset == 16


def test_split_plan(L):
    """The automatic split count minimises waves x (split length + 3), is capped by
    the kv tiles, never leaves a split empty, and sizes the fp32 parts of O and
    LSE.  Expected counts worked by hand over every candidate."""
    # 64 units, 256 kv tiles: n = 7 -> 37 tiles, 448 units = 3 waves, cost 120;
    # n = 3: 2 waves of 89; n = 6: 3 waves of 46; n = 14: 6 waves of 22
    assert L.fa_fwd_split_count(1, 16, 1024, 32768, 152) == 7
    assert L.fa_fwd_split_count(1, 16, 16384, 16384, 152) == 1  # enough units already
    # 16 units, 128 kv tiles: n = 9 -> 15 tiles, 144 units in one wave, cost 18
    assert L.fa_fwd_split_count(2, 8, 128, 16384, 152) == 9
    assert L.fa_fwd_split_count(1, 1, 1, 300, 152) == 3         # only 3 kv tiles
    assert L.fa_fwd_split_count(0, 16, 1024, 32768, 152) == 0   # invalid sizes
    assert L.fa_fwd_split_count(1, 16, 1024, 0, 152) == 0
    # 5 requested over 256 kv tiles: 52 per split, 5 splits; 16 * 1024 rows
    rows = 16 * 1024
    assert L.fa_fwd_split_workspace_bytes(1, 16, 1024, 32768, 128, 5) == 5 * rows * (128 + 1) * 4
    # 7 requested over 3 kv tiles: 3 splits; 1600 rows at D = 64
    assert L.fa_fwd_split_workspace_bytes(1, 16, 100, 300, 64, 7) == 3 * 1600 * (64 + 1) * 4
    # 4 requested over 10 kv tiles: 3 per split -> 4 splits; 3 requested: 4 per split -> 3
    assert L.fa_fwd_split_workspace_bytes(1, 1, 128, 1280, 64, 4) == 4 * 128 * 65 * 4
    assert L.fa_fwd_split_workspace_bytes(1, 1, 128, 1280, 64, 3) == 3 * 128 * 65 * 4
    assert L.fa_fwd_split_workspace_bytes(1, 16, 1024, 32768, 128, 1) == 0  # no split
    assert L.fa_fwd_split_workspace_bytes(1, 16, 1024, 32768, 96, 5) == 0   # bad D


def test_split_validation(L):
    def split(n=3, ws=P16, wsb=1 << 30, q=P16, Sq=256, mod=None):
        return L.fa_fwd_split(q, P16, P16, P16, P16, 1, 2, 2, Sq, 1024, 64, mod, 0.125, n, ws,
                              wsb, None)
    assert split(n=-1) == 1
    assert split(q=None) == 1
    assert split(q=P17) == 3
    assert split(Sq=0, q=None) == 0  # nothing to do
    bad = fa.ScoreMod(-1, -1, None, 16 * 1024 + 2)  # misaligned key counts
    assert split(mod=ctypes.byref(bad)) == 3


def test_merge_validation(L):
    def merge(op=P16, lp=P16, n=2, o=P16, lse=P16, rows=10, D=128):
        return L.fa_lse_merge(op, lp, n, o, lse, rows, D, None)
    assert merge(rows=0, op=None, lp=None, o=None, lse=None) == 0
    assert merge(n=0) == 1
    assert merge(rows=-1) == 1
    assert merge(D=96) == 2
    assert merge(op=None) == 1
    assert merge(op=P17) == 3
    assert merge(o=ctypes.c_void_p(16 * 1024 + 8)) == 3
    assert merge(lp=ctypes.c_void_p(16 * 1024 + 2)) == 3


def test_wait_hook_validation(L):
    assert L.fa_wait_test(P16, 2, P16, None) == 1    # unknown wait
    assert L.fa_wait_test(None, 0, P16, None) == 1   # the semaphore wait needs its flag
    assert L.fa_wait_test(P16, 0, None, None) == 1   # no status word
    assert L.fa_wait_test(ctypes.c_void_p(16 * 1024 + 2), 0, P16, None) == 3
    assert L.fa_wait_test(None, 1, ctypes.c_void_p(16 * 1024 + 1), None) == 3


def test_exp2_hook_validation(L):
    assert L.fa_exp2_test(None, None, 0, 0, None) == 0
    assert L.fa_exp2_test(None, None, -1, 0, None) == 1
    assert L.fa_exp2_test(P16, P16, 4, 3, None) == 1
    assert L.fa_exp2_test(P16, P16, 4, -1, None) == 1


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.fwd(x, x, x)


def test_python_binding_checks_score_mod_arrays():
    """The slopes and key counts must be device arrays of the right type and
    length; the binding refuses anything else before calling the library."""
    import torch
    counts = torch.tensor([3, 4], dtype=torch.int32)  # host memory
    with pytest.raises(TypeError):
        fa._score_mod(False, None, None, 2, counts, 2)
    with pytest.raises(TypeError):
        fa._score_mod(False, (-1, 0), torch.zeros(2), 2)
    with pytest.raises(ValueError):
        fa._score_mod(True, (-1, 0), None, 2)  # the causal flag and a window together
    # nothing to modify: the plain entry points apply
    assert fa._score_mod(True, None, None, 2) is None


def test_bwd_kernel_switch(L):
    prev = ctypes.c_int(-1)
    assert L.fa_set_bwd_kernel(2, ctypes.byref(prev)) == 0
    assert prev.value == 0  # the default: automatic choice
    assert L.fa_set_bwd_kernel(7, ctypes.byref(prev)) == 1  # rejected, nothing changes
    assert L.fa_set_bwd_kernel(1, None) == 0
    assert L.fa_set_bwd_kernel(0, ctypes.byref(prev)) == 0
    assert prev.value == 1
