"""The C-ABI library without a GPU: it loads, exports every symbol that
include/fa.h declares, rejects bad arguments with the documented status codes
before touching any device, and its host-side split arithmetic is consistent.
"""
import os
import re

import pytest

from attention_forward_prefill_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "fa_prefill" in names and "fa_decode" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding._SIGNATURES) >= set(names)


def declarations():
    """{name: (return type, [parameter declarations])} from include/fa.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(fa_\w+)\s*\(([^)]*)\)\s*;", text):
        ret = re.sub(r"\s+", " ", m.group(1)).replace(" *", "*").strip()
        params = [re.sub(r"\s+", " ", x).replace(" *", "* ").replace("* ", "*").strip()
                  for x in m.group(3).split(",")]
        out[m.group(2)] = (ret, params)
    return out


# The boundary's entry points, call for call, with their parameter lists.
BOUNDARY = {
    "fa_prefill": ("int", ["const void*q", "const void*k", "const void*v", "void*out", "int B",
                           "int H", "int N", "int d", "int causal", "float scale", "void*stream"]),
    "fa_prefill_ex": ("int", ["const void*q", "const void*k", "const void*v", "void*out", "int B",
                              "int H", "int N", "int d", "int causal", "float scale",
                              "fa_dtype in_dtype", "fa_dtype out_dtype", "void*stream"]),
    "fa_decode": ("int", ["const void*q", "const void*k_cache", "const void*v_cache",
                          "const int32_t*seq_lens", "void*out", "int B", "int H", "int max_len",
                          "int d", "float scale", "void*stream"]),
    "fa_decode_ex": ("int", ["const void*q", "const void*k_cache", "const void*v_cache",
                             "const int32_t*seq_lens", "void*out", "int B", "int H", "int max_len",
                             "int d", "float scale", "fa_dtype in_dtype", "fa_dtype out_dtype",
                             "int num_splits", "void*workspace", "size_t workspace_bytes",
                             "void*stream"]),
    "fa_decode_choose_splits": ("int", ["int B", "int H", "int max_len", "int device"]),
    "fa_decode_workspace_bytes": ("size_t", ["int B", "int H", "int max_len", "int d",
                                             "int num_splits"]),
    "fa_status_string": ("const char*", ["int status"]),
    "fa_last_cuda_error": ("int", ["void"]),
}


def test_header_matches_the_boundary_call_for_call():
    decl = declarations()
    for name, (ret, params) in BOUNDARY.items():
        assert name in decl, name
        assert decl[name] == (ret, params), (name, decl[name])
    text = open(HEADER).read()
    want = ["FA_OK = 0", "FA_ERR_NULL = 1", "FA_ERR_SHAPE = 2", "FA_ERR_HEAD_DIM = 3",
            "FA_ERR_DTYPE = 4", "FA_ERR_ALIGN = 5", "FA_ERR_SCALE = 6", "FA_ERR_ARCH = 7",
            "FA_ERR_WORKSPACE = 8", "FA_ERR_CUDA = 9", "FA_ERR_WATCHDOG = 10",
            "FA_ERR_SEQ_LEN = 11"]
    for w in want:
        assert w in text, w
    assert "FA_F16 = 0, FA_BF16 = 1, FA_F32 = 2" in text
    for code, name in binding.STATUS_NAMES.items():
        assert f"{name} = {code}" in text


def test_diagnostic_calls_check_arguments_first(lib):
    assert binding.fa_watchdog_selftest(1_000_000, None, None) == binding.FA_ERR_NULL
    assert binding.fa_watchdog_selftest(1_000_000, A + 4, None) == binding.FA_ERR_ALIGN
    assert binding.fa_watchdog_selftest(10, A, None) == binding.FA_ERR_SHAPE
    assert binding.fa_watchdog_selftest(2_000_000_000, A, None) == binding.FA_ERR_SHAPE
    assert binding.fa_read_probe(None, 16, A, None) == binding.FA_ERR_NULL
    assert binding.fa_read_probe(A + 8, 16, A, None) == binding.FA_ERR_ALIGN
    assert binding.fa_read_probe(A, 16, A + 2, None) == binding.FA_ERR_ALIGN
    assert binding.fa_read_probe(A, 0, A, None) == binding.FA_ERR_SHAPE
    assert binding.fa_read_probe(A, 24, A, None) == binding.FA_ERR_SHAPE
    assert binding.load().fa_pool_stats(None, 0) == binding.FA_ERR_NULL


def test_status_strings_and_version(lib):
    for code in range(14):
        assert binding.status_string(code) != "unknown status"
    assert binding.status_string(999) == "unknown status"
    assert binding.fa_version() >= 20100  # 2.1: fa_prefill_backward_ex


A = 1 << 20   # an aligned fake address: validation must reject before using it
B_ = 1 << 28


@pytest.mark.parametrize("args,status", [
    ((None, A, A, B_, 1, 1, 1, 64, 0, 1.0, 0, 0), 1),
    ((A, A, A, B_, 0, 1, 1, 64, 0, 1.0, 0, 0), 2),
    ((A, A, A, B_, 1, 1, -3, 64, 0, 1.0, 0, 0), 2),
    ((A, A, A, B_, 65536, 65536, 2, 64, 0, 1.0, 0, 0), 2),
    ((A, A, A, B_, 1, 1, 1, 96, 0, 1.0, 0, 0), 3),
    ((A, A, A, B_, 1, 1, 1, 64, 0, 1.0, 2, 0), 4),
    ((A, A, A, B_, 1, 1, 1, 64, 0, 1.0, 0, 7), 4),
    ((A + 8, A, A, B_, 1, 1, 1, 64, 0, 1.0, 0, 0), 5),
    ((A, A, A, B_ + 2, 1, 1, 1, 64, 0, 1.0, 0, 0), 5),
    ((A, A, A, B_, 1, 1, 1, 64, 0, float("nan"), 0, 0), 6),
    ((A, A, A, B_, 1, 1, 1, 64, 0, float("inf"), 0, 0), 6),
    ((A, A, A, A, 1, 1, 1, 64, 0, 1.0, 0, 0), binding.FA_ERR_ALIAS),
    ((A, A, A, A + 64, 1, 2, 8, 64, 0, 1.0, 0, 0), binding.FA_ERR_ALIAS),
])
def test_prefill_argument_errors(lib, args, status):
    q, k, v, out, B, H, N, d, causal, scale, it, ot = args
    assert binding.fa_prefill_ex(q, k, v, out, B, H, N, d, causal, scale, it, ot, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, A, A, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 1),
    ((A, A, A, B_, 1, 6, 4, 8, 8, 64, 0, 1.0, 0, 0, 0), 2),      # Hq not a multiple of Hkv
    ((A, A, A, B_, 1, 4, 0, 8, 8, 64, 0, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, 1, 4, 2, 8, 0, 64, 0, 1.0, 0, 0, 0), 2),      # no keys
    ((A, A, A, B_, 1, 4, 2, 0, 8, 64, 0, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 80, 0, 1.0, 0, 0, 0), 3),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 3, 0), 4),
    ((A, A, A + 4, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 5),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 64, 0, float("-inf"), 0, 0, 0), 6),
    ((A, B_ - 64, A, B_, 1, 4, 2, 8, 1024, 64, 0, 1.0, 0, 0, 0), binding.FA_ERR_ALIAS),  # k runs into out
])
def test_gqa_prefill_argument_errors(lib, args, status):
    assert binding.fa_prefill_gqa(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, A, A, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 1),
    ((A, A, A, None, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 1),
    ((A, A, A, B_, 1, 6, 4, 8, 8, 64, 0, 1.0, 0, 0, 0), 2),      # Hq not a multiple of Hkv
    ((A, A, A, B_, 0, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 96, 0, 1.0, 0, 0, 0), 3),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 2, 0, 0), 4),
    ((A, A, A + 8, B_, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), 5),
    ((A, A, A, B_, 1, 4, 2, 8, 8, 64, 0, float("nan"), 0, 0, 0), 6),
    ((A, A, A, A + 256, 1, 4, 2, 8, 8, 64, 0, 1.0, 0, 0, 0), binding.FA_ERR_ALIAS),  # out inside q
])
def test_host_buffer_prefill_argument_errors(lib, args, status):
    # the host-buffer entry point validates like the device one, before any CUDA call
    assert binding.fa_prefill_host(*args, None) == status


CU = 1 << 16


@pytest.mark.parametrize("args,status", [
    ((A, A, A, B_, None, CU, 2, 4, 2, 64, 64, 32, 32, 64, 1, 1.0, 0, 0, 0), 1),
    ((A, A, A, B_, CU + 2, CU, 2, 4, 2, 64, 64, 32, 32, 64, 1, 1.0, 0, 0, 0), 5),
    ((A, A, A, B_, CU, CU, 2, 4, 3, 64, 64, 32, 32, 64, 1, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, CU, CU, 0, 4, 2, 64, 64, 32, 32, 64, 1, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, CU, CU, 2, 4, 2, 64, -1, 32, 32, 64, 1, 1.0, 0, 0, 0), 2),
    ((A, A, A, B_, CU, CU, 2, 4, 2, 64, 64, 32, 32, 100, 1, 1.0, 0, 0, 0), 3),
    ((A, A, A, A, CU, CU, 2, 4, 2, 64, 64, 32, 32, 64, 1, 1.0, 0, 0, 0), binding.FA_ERR_ALIAS),
    # no query rows: nothing to do, and no device is touched
    ((A, A, A, B_, CU, CU, 2, 4, 2, 0, 64, 0, 32, 64, 1, 1.0, 0, 0, 0), 0),
])
def test_varlen_prefill_argument_errors(lib, args, status):
    assert binding.fa_prefill_varlen(*args, None) == status


def test_grouped_decode_argument_errors(lib):
    L = 1 << 24
    base = dict(q=A, k=A, v=A, lens=L, out=B_, B=2, Hq=14, Hkv=2, max_len=4096, d=64, scale=0.125,
                it=0, ot=0, splits=0, ws=None, wsb=0)

    def call(**kw):
        a = {**base, **kw}
        return binding.fa_decode_gqa(a["q"], a["k"], a["v"], a["lens"], a["out"], a["B"], a["Hq"],
                                     a["Hkv"], a["max_len"], a["d"], a["scale"], a["it"], a["ot"],
                                     a["splits"], a["ws"], a["wsb"], None)
    assert call(Hkv=4) == 2           # 14 query heads cannot share 4 cache heads
    assert call(Hkv=0) == 2
    assert call(q=None) == 1
    assert call(d=32) == 3
    assert call(lens=L + 2) == 5
    assert call(splits=4096 // 64 + 1) == binding.FA_ERR_SPLITS
    # 32 query heads per cache head: 4 per CTA, so a chunk may hold 12K rows
    assert call(Hq=32, Hkv=1, max_len=60000, splits=1) == binding.FA_ERR_SPLITS
    assert call(ws=1 << 12, wsb=16, splits=4) == 8


@pytest.mark.parametrize("B,Hq,Hkv,L", [(1, 14, 2, 4096), (32, 14, 2, 4096), (8, 32, 1, 1000),
                                        (4, 8, 8, 4096)])
def test_grouped_split_choice(lib, B, Hq, Hkv, L):
    s = binding.fa_decode_splits_for_sms(B, Hq, Hkv, L, 152)
    rows = Hkv * ((Hq // Hkv + 3) // 4)
    if Hq == Hkv:
        assert s == binding.fa_decode_splits_for_sms(B, Hq, Hq, L, 152)
    else:   # about 5 CTAs per SM, chunks of 64..512 rows, rounded to 64-row chunks
        cdiv = lambda a, b: -(-a // b)
        want = min(max(cdiv(5 * 152, B * rows), cdiv(L, 512)), cdiv(L, 64))
        chunk = cdiv(cdiv(L, want), 64) * 64
        assert s == cdiv(L, chunk)
    assert 1 <= s <= (L + 63) // 64
    assert binding.fa_decode_splits_for_sms(B, Hq, 3, L, 152) < 0 or Hq % 3 == 0


def test_backward_argument_errors(lib):
    args = dict(q=A, k=A + 4096, v=A + 8192, out=A + 12288, dout=A + 16384, lse=A + 20480,
                dq=B_, dk=B_ + (1 << 20), dv=B_ + (2 << 20), B=1, H=6, Hkv=2, N=8, d=64, causal=1,
                scale=0.125, it=0, gt=2)

    def call(**kw):
        a = {**args, **kw}
        return binding.fa_prefill_backward(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"],
                                           a["dq"], a["dk"], a["dv"], a["B"], a["H"], a["Hkv"],
                                           a["N"], a["d"], a["causal"], a["scale"], a["it"], a["gt"],
                                           None)
    assert call(lse=None) == 1
    assert call(Hkv=4) == 2          # 6 query heads cannot share 4 key/value heads
    assert call(N=0) == 2
    assert call(d=96) == 3
    assert call(gt=7) == 4
    assert call(lse=A + 20482) == 5
    assert call(scale=float("nan")) == 6
    assert call(dk=A) == binding.FA_ERR_ALIAS          # dk over q
    assert call(dv=B_ + 16) == binding.FA_ERR_ALIAS    # dv over dq


@pytest.mark.parametrize("flags", [binding.FA_BWD_FLAG_NONE, binding.FA_BWD_RECOMPUTE_DQ, 0x80])
def test_backward_ex_argument_errors_match_the_plain_call(lib, flags):
    # the flags only pick the dQ pass: every argument error is the plain call's
    args = dict(q=A, k=A + 4096, v=A + 8192, out=A + 12288, dout=A + 16384, lse=A + 20480,
                dq=B_, dk=B_ + (1 << 20), dv=B_ + (2 << 20), B=1, H=6, Hkv=2, N=8, d=64, causal=1,
                scale=0.125, it=0, gt=2)
    order = ("q", "k", "v", "out", "dout", "lse", "dq", "dk", "dv", "B", "H", "Hkv", "N", "d", "causal",
             "scale", "it", "gt")
    for bad in (dict(lse=None), dict(Hkv=4), dict(N=0), dict(d=96), dict(gt=7), dict(lse=A + 20482),
                dict(scale=float("nan")), dict(dk=A), dict(dv=B_ + 16), dict(q=A + 8)):
        a = {**args, **bad}
        plain = binding.fa_prefill_backward(*(a[x] for x in order), None)
        ex = binding.fa_prefill_backward_ex(*(a[x] for x in order), flags, None)
        assert plain == ex != binding.FA_OK, bad


def test_plain_prefill_checks_too(lib):
    assert binding.fa_prefill(None, A, A, B_, 1, 1, 1, 64, 0, 1.0, None) == 1
    assert binding.fa_prefill(A, A, A, B_, 1, 1, 1, 80, 0, 1.0, None) == 3


S = 1 << 24  # seq_lens


@pytest.mark.parametrize("kw,status", [
    (dict(seq_lens=None), 1),
    (dict(B=0), 2),
    (dict(d=32), 3),
    (dict(in_dtype=2), 4),
    (dict(q=A + 4), 5),
    (dict(seq_lens=S + 2), 5),
    (dict(workspace=A + 8, workspace_bytes=1 << 20), 5),
    (dict(scale=float("nan")), 6),
    (dict(num_splits=-1), binding.FA_ERR_SPLITS),
    (dict(num_splits=65), binding.FA_ERR_SPLITS),
    (dict(num_splits=4, workspace=1 << 30, workspace_bytes=16), 8),
    (dict(out=S), binding.FA_ERR_ALIAS),
])
def test_decode_argument_errors(lib, kw, status):
    a = dict(q=A, k=1 << 26, v=1 << 27, seq_lens=S, out=B_, B=2, H=3, max_len=4096, d=64,
             scale=0.125, in_dtype=0, out_dtype=0, num_splits=0, workspace=None,
             workspace_bytes=0)
    a.update(kw)
    got = binding.fa_decode_ex(a["q"], a["k"], a["v"], a["seq_lens"], a["out"], a["B"], a["H"],
                               a["max_len"], a["d"], a["scale"], a["in_dtype"], a["out_dtype"],
                               a["num_splits"], a["workspace"], a["workspace_bytes"], None)
    assert got == status


@pytest.mark.parametrize("B,H,L,sms", [(1, 14, 4096, 152), (8, 14, 4096, 152), (32, 14, 4096, 152),
                                       (1, 12, 4096, 148), (3, 2, 1000, 152), (1, 1, 1, 152),
                                       (2, 2, 100000, 152), (64, 64, 4096, 152)])
def test_split_choice_host_logic(lib, B, H, L, sms):
    s = binding.fa_decode_splits_for_sms(B, H, H, L, sms)
    assert s >= 1
    chunk = binding.fa_decode_chunk_len(L, s)
    assert chunk % 64 == 0
    assert chunk * s >= L and (s - 1) * chunk < L          # every row in exactly one chunk
    assert chunk <= 512                                     # no CTA longer than 512 rows
    # target: about three CTAs per SM over the whole (b, h, chunk) grid, at
    # least one chunk per 512 rows, at most one per 64 rows
    target = min(max(-(-3 * sms // (B * H)), -(-L // 512), 1), -(-L // 64))
    assert s <= target
    assert chunk == 64 or -(-L // (chunk - 64)) > target    # chunk is the smallest that fits
    ws = binding.fa_decode_workspace_bytes(B, H, L, 64, s)
    assert ws >= B * H * s * (64 + 2) * 4


def test_split_choice_bad_args(lib):
    assert binding.fa_decode_choose_splits(0, 1, 10, 0) == -binding.FA_ERR_SHAPE
    assert binding.fa_decode_splits_for_sms(0, 1, 1, 10, 152) == -binding.FA_ERR_SHAPE
    assert binding.fa_decode_splits_for_sms(1, 1, 1, 10, 0) == -binding.FA_ERR_SHAPE
    assert binding.fa_decode_chunk_len(0, 1) < 0
    assert binding.fa_decode_workspace_bytes(1, 1, 10, 48, 1) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load()
