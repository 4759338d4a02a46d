"""The C ABI without a GPU: the library builds and loads, exports every
function include/satk.h declares, maps status codes, sizes the rescue
scratch, and rejects invalid arguments before launching anything.

Calls here never reach a kernel: each passes arguments that the host checks
refuse.  They use placeholder (never dereferenced) pointers, so they only
run where no GPU is present; tests/test_gpu_parity.py repeats them with real
device buffers."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from sparse_attention_indexer_radix_gb300 import binding
from sparse_attention_indexer_radix_gb300 import build as satk_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "satk.h")

EINVAL, EUNSUPPORTED = -1, -2
no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="placeholder pointers only where no GPU can run a kernel")


@pytest.fixture(scope="module")
def lib():
    satk_build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\(", text,
                                 flags=re.M)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"satk_topk_rows", "satk_dcp_pack", "satk_dcp_merge_select",
            "satk_dcp_rescue_select", "satk_rescue_recv_words", "satk_status_string",
            "topk_rows", "dcp_pack", "dcp_merge_select", "dcp_rescue_select",
            "satk_dcp_topk_pack", "dcp_topk_pack"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} is declared in satk.h but not exported"
    assert set(binding.EXPORTS) <= set(names)


def test_status_strings_and_recv_words(lib):
    assert lib.satk_status_string(0) == b"ok"
    for rc in (-1, -2, -3, 99):
        assert len(lib.satk_status_string(rc)) > 0
    assert lib.satk_rescue_recv_words(128, 384, 2048) == 128 * 5 * (2048 + 64)
    assert lib.satk_rescue_recv_words(3, 64, 512) == 3 * 7 * (512 + 16)
    assert lib.satk_rescue_recv_words(-1, 64, 512) == 0


P = ctypes.c_void_p(4096)  # placeholder: never dereferenced by a rejected call
NULL = None


@no_gpu
@pytest.mark.parametrize("name", ["satk_topk_rows", "satk_topk_rows_sorted"])
def test_topk_rows_rejects(lib, name):
    f = getattr(lib, name)
    ok = dict(x=P, dt=0, rows=4, cols=100, ld=100, re=NULL, k=8, out=P, ldo=8)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["x"], a["dt"], a["rows"], a["cols"], a["ld"], a["re"], a["k"], a["out"],
                 a["ldo"], NULL)
    assert call(x=NULL) == EINVAL
    assert call(out=NULL) == EINVAL
    assert call(rows=-1) == EINVAL
    assert call(cols=-1) == EINVAL
    assert call(ld=99) == EINVAL
    assert call(k=0) == EINVAL
    assert call(k=4097, ldo=5000) == EINVAL
    assert call(ldo=7) == EINVAL
    assert call(dt=2) == EINVAL
    assert call(cols=2**31, ld=2**31) == EINVAL
    assert call(rows=0) == 0  # nothing to do, nothing launched


@no_gpu
def test_pack_rejects(lib):
    f = lib.satk_dcp_pack
    ok = dict(lg=P, rows=4, S=100, ld=100, li=P, ldi=64, n=64, re=NULL, out=P)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["lg"], a["rows"], a["S"], a["ld"], a["li"], a["ldi"], a["n"], a["re"],
                 a["out"], NULL)
    assert call(lg=NULL) == EINVAL
    assert call(li=NULL) == EINVAL
    assert call(out=NULL) == EINVAL
    assert call(n=48, ldi=48) == EINVAL
    assert call(n=0, ldi=0) == EINVAL
    assert call(ldi=63) == EINVAL
    assert call(ld=99) == EINVAL
    assert call(rows=0) == 0


@no_gpu
def test_topk_pack_rejects(lib):
    f = lib.satk_dcp_topk_pack
    ok = dict(lg=P, rows=4, S=100, ld=100, re=NULL, n=64, out=P)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["lg"], a["rows"], a["S"], a["ld"], a["re"], a["n"], a["out"], NULL)
    assert call(lg=NULL) == EINVAL
    assert call(out=NULL) == EINVAL
    assert call(rows=-1) == EINVAL
    assert call(S=-1) == EINVAL
    assert call(ld=99) == EINVAL
    assert call(n=48) == EINVAL
    assert call(n=0) == EINVAL
    assert call(n=4096 + 32) == EINVAL
    assert call(S=2**31, ld=2**31) == EINVAL
    assert call(rows=0) == 0


@no_gpu
def test_merge_rejects(lib):
    f = lib.satk_dcp_merge_select
    ok = dict(c=P, fmt=1, W=8, T=4, n=384, k=2048, ids=P, ldo=2048, sat=NULL, st=NULL)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["c"], a["fmt"], a["W"], a["T"], a["n"], a["k"], a["ids"], a["ldo"],
                 a["sat"], a["st"], NULL)
    assert call(c=NULL) == EINVAL
    assert call(ids=NULL) == EINVAL
    assert call(W=0) == EINVAL
    assert call(W=17) == EINVAL          # packed: at most 16 ranks
    assert call(n=100) == EINVAL         # n % 32
    assert call(k=0) == EINVAL
    assert call(ldo=2047) == EINVAL
    assert call(fmt=7) == EINVAL
    assert call(fmt=0, sat=P) == EINVAL  # no saturation word for pairs
    assert call(fmt=0, W=32, n=2048) == EUNSUPPORTED
    assert call(T=0) == 0


@no_gpu
def test_rescue_rejects(lib):
    f = lib.satk_dcp_rescue_select
    ok = dict(p=P, W=8, T=4, n=384, k=2048, lg=P, S=1000, ld=1000, re=NULL, sat=P, recv=P,
              ids=P, ldo=2048, st=NULL)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["p"], a["W"], a["T"], a["n"], a["k"], a["lg"], a["S"], a["ld"], a["re"],
                 a["sat"], a["recv"], a["ids"], a["ldo"], a["st"], NULL)
    for name in ("p", "lg", "sat", "recv", "ids"):
        assert call(**{name: NULL}) == EINVAL
    assert call(W=17) == EINVAL
    assert call(n=2048) == EINVAL        # n must be below k
    assert call(k=2000, ldo=2048) == EINVAL
    assert call(k=8192, ldo=8192) == EINVAL
    assert call(ld=999) == EINVAL
    assert call(W=16, n=128, k=4096, ldo=4096) == EUNSUPPORTED
    assert call(T=0) == 0


def test_binding_refuses_cpu_tensors():
    x = torch.zeros((2, 8))
    with pytest.raises(binding.SatkError):
        binding.topk_rows(x, 2)


@no_gpu
def test_emit_rows_rejects(lib):
    f = lib.satk_dcp_emit_rows
    ok = dict(ids=P, T=4, k=64, ld=64, W=8, rank=3, req=P, table=P, R=2, ldt=16, maxb=16,
              B=64, stride=64, rows=P, ldr=64, valid=P, st=NULL)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["ids"], a["T"], a["k"], a["ld"], a["W"], a["rank"], a["req"], a["table"],
                 a["R"], a["ldt"], a["maxb"], a["B"], a["stride"], a["rows"], a["ldr"],
                 a["valid"], a["st"], NULL)
    for name in ("ids", "req", "table", "rows", "valid"):
        assert call(**{name: NULL}) == EINVAL
    assert call(T=-1) == EINVAL
    assert call(k=0) == EINVAL
    assert call(ld=63) == EINVAL
    assert call(W=0) == EINVAL
    assert call(rank=8) == EINVAL
    assert call(rank=-1) == EINVAL
    assert call(R=-1) == EINVAL
    assert call(maxb=17) == EINVAL    # wider than the table's row stride
    assert call(B=0) == EINVAL
    assert call(ldr=63) == EINVAL
    assert call(T=0) == 0             # nothing to do, nothing launched
