"""The C ABI: the library builds for sm_103a, exports every declared symbol,
and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import exact_attention_17_gb300 as fa2
from exact_attention_17_gb300 import build as libbuild

HEADER = os.path.join(libbuild.INCLUDE, "fa2.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return fa2.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa2_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "fa2_forward" in names and "fa2_status_string" in names
    assert set(names) == set(fa2.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(12):
        s = fa2.fa2_status_string(code)
        assert s and s != "unknown status"
    assert fa2.fa2_status_string(12345) == "unknown status"


def call(**kw):
    args = dict(Q=16, K=16, V=16, O=16, LSE=16, B=1, H=1, Nq=8, Nk=8, d=64, causal=0,
                scale=0.125, stream=None)
    args.update(kw)
    return fa2.fa2_forward(args["Q"], args["K"], args["V"], args["O"], args["LSE"], args["B"],
                           args["H"], args["Nq"], args["Nk"], args["d"], args["causal"],
                           args["scale"], args["stream"])


def _split_static(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, stream, num_splits=4):
    return fa2.fa2_forward_splitkv_static(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale,
                                          num_splits, stream)


def _split_workspace(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, stream, num_splits=4):
    return fa2.fa2_forward_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, num_splits,
                                   256, 1 << 20, stream)


FORWARD_ENTRY_POINTS = {"fa2_forward": lambda: fa2.fa2_forward,
                        "fa2_forward_simt": lambda: fa2.fa2_forward_simt,
                        "fa2_forward_splitkv": lambda: _split_workspace,
                        "fa2_forward_splitkv_static": lambda: _split_static}


@pytest.mark.parametrize("fn", sorted(FORWARD_ENTRY_POINTS))
def test_host_side_argument_errors(lib, fn):
    f = FORWARD_ENTRY_POINTS[fn]()

    def c(**kw):
        a = dict(Q=16, K=16, V=16, O=16, LSE=16, B=1, H=1, Nq=8, Nk=8, d=64, causal=0,
                 scale=0.125, stream=None)
        a.update(kw)
        return f(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["Nq"], a["Nk"],
                 a["d"], a["causal"], a["scale"], a["stream"])

    # empty problems are valid and launch nothing
    assert c(B=0) == fa2.FA2_OK
    assert c(H=0, Q=None) == fa2.FA2_OK
    assert c(Nq=0) == fa2.FA2_OK
    # sizes
    assert c(B=-1) == fa2.FA2_ERR_SHAPE
    assert c(Nk=-1) == fa2.FA2_ERR_SHAPE
    assert c(Nk=0) == fa2.FA2_ERR_SHAPE
    assert c(B=1 << 16, H=1 << 16) == fa2.FA2_ERR_SHAPE
    for d in (0, 32, 96, 192, 512):
        assert c(d=d) == fa2.FA2_ERR_HEADDIM
    for s in (0.0, -1.0, float("inf"), float("nan")):
        assert c(scale=s) == fa2.FA2_ERR_SCALE
    # head dimension 256 passes the head-dimension check (the scale check comes next)
    assert c(d=256, scale=0.0) == fa2.FA2_ERR_SCALE
    for name in ("Q", "K", "V", "O", "LSE"):
        assert c(**{name: None}) == fa2.FA2_ERR_NULL
    for name in ("Q", "K", "V", "O"):
        assert c(**{name: 24}) == fa2.FA2_ERR_ALIGN
    assert c(LSE=18) == fa2.FA2_ERR_ALIGN


@pytest.mark.parametrize("fn", [_split_static, _split_workspace])
def test_split_entry_points_check_the_split_count_first(lib, fn):
    args = (16, 16, 16, 16, 16, 1, 1, 8, 8, 64, 0, 0.125, None)
    for n in (0, -1, 65, 1000):
        assert fn(*args, num_splits=n) == fa2.FA2_ERR_SHAPE
    # a valid count on an empty problem launches nothing
    empty = (16, 16, 16, 16, 16, 0, 1, 8, 8, 64, 0, 0.125, None)
    assert fn(*empty, num_splits=64) == fa2.FA2_OK
    assert fn(*empty, num_splits=1) == fa2.FA2_OK


def test_typed_entry_point_rejects_bad_element_types_on_the_host(lib):
    args = (16, 16, 16, 16, 16, 1, 1, 8, 8, 64, 0, 0.125)
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_FP32, fa2.FA2_DTYPE_FP32, None) == fa2.FA2_ERR_DTYPE
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_BF16, fa2.FA2_DTYPE_FP16, None) == fa2.FA2_ERR_DTYPE
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_FP16, fa2.FA2_DTYPE_BF16, None) == fa2.FA2_ERR_DTYPE
    # valid types, empty problem: nothing launched
    empty = (16, 16, 16, 16, 16, 0, 1, 8, 8, 64, 0, 0.125)
    assert fa2.fa2_forward_typed(*empty, fa2.FA2_DTYPE_FP16, fa2.FA2_DTYPE_FP16, None) == fa2.FA2_OK


def test_backward_workspace_bytes(lib):
    # two [B*H][ceil(Nq/128)*128] fp32 arrays, each rounded up to 256 bytes
    assert fa2.fa2_backward_workspace_bytes(1, 1, 1) == 2 * 512
    assert fa2.fa2_backward_workspace_bytes(2, 3, 200) == 2 * 6 * 256 * 4
    assert fa2.fa2_backward_workspace_bytes(1, 1, 0) == 0
    assert fa2.fa2_backward_workspace_bytes(-1, 1, 8) == 0


def test_backward_host_side_argument_errors(lib):
    def c(**kw):
        a = dict(Q=16, K=16, V=16, O=16, dO=16, LSE=16, dQ=16, dK=16, dV=16, B=1, H=1, Nq=8, Nk=8,
                 d=64, causal=0, scale=0.125, ws=256, wss=1 << 20)
        a.update(kw)
        return fa2.fa2_backward(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["LSE"], a["dQ"], a["dK"],
                                a["dV"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["causal"],
                                a["scale"], a["ws"], a["wss"], None)

    # empty problems launch nothing
    assert c(B=0) == fa2.FA2_OK
    assert c(Nq=0, Nk=0) == fa2.FA2_OK
    # sizes
    assert c(Nq=-1) == fa2.FA2_ERR_SHAPE
    assert c(Nk=0) == fa2.FA2_ERR_SHAPE
    for d in (0, 32, 96, 256):   # the backward kernels cover 64 and 128
        assert c(d=d) == fa2.FA2_ERR_HEADDIM
    for s in (0.0, -1.0, float("inf"), float("nan")):
        assert c(scale=s) == fa2.FA2_ERR_SCALE
    for name in ("Q", "K", "V", "O", "dO", "LSE", "dQ", "dK", "dV", "ws"):
        assert c(**{name: None}) == fa2.FA2_ERR_NULL
    # with no query rows only dK and dV are needed
    assert c(Nq=0, dK=None) == fa2.FA2_ERR_NULL
    for name in ("Q", "K", "V", "O", "dO", "dQ", "dK", "dV"):
        assert c(**{name: 24}) == fa2.FA2_ERR_ALIGN
    assert c(LSE=18) == fa2.FA2_ERR_ALIGN
    assert c(ws=272) == fa2.FA2_ERR_ALIGN


def test_splitkv_workspace_and_merge_head_dims(lib):
    # O_part [S][rows][d] fp32 then LSE_part [S][rows], each rounded up to 256 bytes
    assert fa2.fa2_splitkv_workspace_bytes(1, 2, 100, 256, 3) == 3 * 200 * 256 * 4 + 2560
    assert fa2.fa2_splitkv_workspace_bytes(1, 2, 100, 96, 3) == 0
    # merge: head dimension checked before the pointers
    assert fa2.fa2_merge(None, None, 2, 8, 96, None, None, None) == fa2.FA2_ERR_HEADDIM
    assert fa2.fa2_merge(None, None, 2, 8, 256, None, None, None) == fa2.FA2_ERR_NULL


def test_fast_division_method():
    """The multiply-and-shift division the forward kernel uses to decode its
    work item (divisors fixed per launch): with l = ceil(log2 d),
    m = ceil(2^(31+l) / d) and s = 31 + l, (n m) >> s == n // d for every
    0 <= n < 2^31 (Granlund and Montgomery 1994).  Checked on the divisors
    where the rounding excess is largest and on the numerators nearest to a
    multiple of d and to 2^31."""
    import random

    def magic(d):
        l = (d - 1).bit_length()
        m = -(-(1 << (31 + l)) // d)
        assert m < 1 << 32
        return m, 31 + l

    rng = random.Random(7)
    divisors = list(range(1, 600)) + [2 ** k + e for k in range(1, 31) for e in (-1, 0, 1)
                                      if 1 <= 2 ** k + e < 2 ** 31]
    divisors += [rng.randrange(1, 2 ** 31) for _ in range(300)] + [2 ** 31 - 1]
    for d in divisors:
        m, s = magic(d)
        ns = {0, 1, d - 1, d, d + 1, 2 ** 31 - 1, 2 ** 31 - 2}
        top = (2 ** 31 - 1) // d * d
        ns |= {top - 1, top, top + d - 1} | {rng.randrange(0, 2 ** 31) for _ in range(40)}
        for n in ns:
            if 0 <= n < 2 ** 31:
                assert (n * m) >> s == n // d, (n, d)


def test_wait_check_rejects_out_of_range_limits_on_the_host(lib):
    for t in (0, 999, 10_000_000_001):
        assert fa2.fa2_check_wait_timeout(t) == fa2.FA2_ERR_SHAPE


def test_typed_backward_rejects_bad_element_types_on_the_host(lib):
    args = [16] * 9 + [1, 1, 8, 8, 64, 0, 0.125]
    for t in (fa2.FA2_DTYPE_FP32, 7, -1):
        assert fa2.fa2_backward_typed(*args, t, 256, 1 << 20, None) == fa2.FA2_ERR_DTYPE
    # valid type, empty problem: nothing launched
    empty = [16] * 9 + [0, 1, 8, 8, 64, 0, 0.125]
    assert fa2.fa2_backward_typed(*empty, fa2.FA2_DTYPE_FP16, 256, 1 << 20, None) == fa2.FA2_OK


def test_recommended_splits_fill_the_gpu(lib):
    """Host arithmetic with a given SM count (152 on GB300)."""
    rec = fa2.fa2_splitkv_recommended_splits
    # grids that already fill the GPU keep one key range
    assert rec(1, 32, 16384, 16384, 152) == 1
    assert rec(4, 16, 4096, 4096, 152) == 1
    assert rec(16, 32, 128, 8192, 152) == 1
    # 2 x 8 heads x 8 query blocks = 128 CTAs on 304 slots, 8 key tiles: the
    # fixed cost of a CTA and the merge outweigh halving the tiles (measured slower)
    assert rec(2, 8, 1000, 1000, 152) == 1
    # one query row per head, 16 heads, 64 key tiles: ranges of four tiles fill one wave
    assert rec(2, 8, 1, 8192, 152) == 16
    # 128 CTAs, 64 key tiles: ranges of 32 tiles in one wave
    assert rec(2, 8, 1000, 8192, 152) == 2
    # never more ranges than key tiles, never more than 64
    assert rec(1, 1, 1, 100, 152) == 1
    assert 1 <= rec(1, 1, 1, 1 << 20, 152) <= 64
    # empty and invalid problems
    assert rec(0, 8, 1000, 1000, 152) == 1
    assert rec(1, 1, 0, 1000, 152) == 1
    assert rec(-1, 1, 10, 10, 152) == 1


def test_host_buffer_entry_point_checks_on_the_host(lib):
    def c(chunks=4, B=1, **kw):
        a = dict(Qh=16, Kh=16, Vh=16, Oh=16, Lh=16, Qd=16, Kd=16, Vd=16, Od=16, Ld=16)
        a.update(kw)
        return fa2.fa2_forward_host(a["Qh"], a["Kh"], a["Vh"], a["Oh"], a["Lh"], a["Qd"], a["Kd"], a["Vd"],
                                    a["Od"], a["Ld"], B, 2, 8, 8, 64, 0, 0.125, chunks, None)

    for n in (0, -3, 17):
        assert c(chunks=n) == fa2.FA2_ERR_SHAPE
    # empty problem: nothing copied or launched
    assert c(B=0, Qh=None) == fa2.FA2_OK
    # the device buffers are checked like fa2_forward's pointers
    assert c(Qd=None) == fa2.FA2_ERR_NULL
    assert c(Od=24) == fa2.FA2_ERR_ALIGN
