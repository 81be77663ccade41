"""The C library's host side, without a GPU: symbols, struct layout, argument checks.

Every call here fails validation before anything touches the CUDA runtime,
or (the decode workspace size) only asks the runtime for the SM count and
falls back to a fixed count without a device, so none of these tests needs
a device.
"""

import ctypes
import os
import subprocess
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def abi():
    from exact_attention_12_gb300 import build, _abi
    if not os.path.exists(build.LIB_PATH):
        build.build()
    return _abi


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function(abi):
    lib = abi.lib()
    declared = _declared_functions()
    assert declared, "no functions found in include/attn.h"
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(declared) == sorted(abi.EXPORTS), (declared, sorted(abi.EXPORTS))


def test_params_struct_layout(abi, tmp_path):
    # the ctypes mirror against the C compiler's layout of include/attn.h
    p = abi.AttnParams
    names = [f[0] for f in p._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "attn.h"', 'int main(void) {',
             '  printf("size %zu\\n", sizeof(attn_params));']
    lines += [f'  printf("{n} %zu\\n", offsetof(attn_params, {n}));' for n in names]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.check_call(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    assert int(got["size"]) == ctypes.sizeof(p) == 144
    for n in names:
        assert int(got[n]) == getattr(p, n).offset, n


def _params(abi, **kw):
    p = abi.AttnParams()
    p.B, p.H, p.N, p.d = 2, 3, 256, 64
    p.dtype = abi.ATTN_BF16
    p.scale = 0.125
    p.stride_b, p.stride_h, p.stride_n = 3 * 256 * 64, 256 * 64, 64
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value,status", [
    ("d", 96, 2), ("d", 32, 2), ("B", -1, 1), ("scale", 0.0, 1), ("scale", -1.0, 1),
    ("scale", float("inf"), 1), ("dropout_p", 1.0, 1), ("dropout_p", -0.1, 1),
    ("philox_offset", 1 << 32, 1), ("stride_n", 60, 1), ("stride_h", 0, 1), ("dtype", 7, 1),
    ("H_kv", 2, 1), ("H_kv", -1, 1), ("H_kv", 1, 1), ("reserved", 1, 1), ("kv_stride_n", 60, 1),
])
def test_invalid_arguments_are_rejected_on_the_host(abi, field, value, status):
    lib = abi.lib()
    p = _params(abi, **{field: value})
    assert lib.attn_workspace_size(ctypes.byref(p), 0) == 0
    fake = ctypes.c_void_p(0x1000)
    st = lib.attn_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, 1 << 20, None)
    assert st == status, lib.attn_last_error()
    assert lib.attn_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(d=64), 2), (dict(d=128, dropout_p=0.1), 2), (dict(d=128, q_descale=-1.0), 1),
    (dict(d=128, v_descale=float("nan")), 1), (dict(d=128, stride_n=136), 1),
    (dict(d=128, reserved2=1), 1),
])
def test_fp8_forward_options_checked_on_the_host(abi, kw, status):
    lib = abi.lib()
    base = dict(dtype=abi.ATTN_FP8_E4M3, stride_b=3 * 256 * 128, stride_h=256 * 128,
                stride_n=128)
    base.update(kw)
    p = _params(abi, **base)
    fake = ctypes.c_void_p(0x1000)
    st = lib.attn_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, 1 << 30, None)
    assert st == status, lib.attn_last_error()


def test_fp8_workspace_holds_the_transposed_values(abi):
    lib = abi.lib()
    p = _params(abi, dtype=abi.ATTN_FP8_E4M3, d=128, N=200, stride_b=3 * 200 * 128,
                stride_h=200 * 128, stride_n=128)
    # header + V^T [B * H][d][256 keys] bytes
    assert lib.attn_workspace_size(ctypes.byref(p), 0) == 256 + 2 * 3 * 128 * 256
    assert lib.attn_workspace_size(ctypes.byref(p), 1) == 0       # no fp8 backward


def test_fp32_backward_is_unsupported(abi):
    lib = abi.lib()
    p = _params(abi, dtype=abi.ATTN_FP32)
    fake = ctypes.c_void_p(0x1000)
    st = lib.attn_bwd(ctypes.byref(p), *([fake] * 10), 1 << 30, None)
    assert st == abi.ATTN_ERR_UNSUPPORTED


def test_workspace_size_and_checks(abi):
    lib = abi.lib()
    p = _params(abi)
    fwd = lib.attn_workspace_size(ctypes.byref(p), 0)
    bwd = lib.attn_workspace_size(ctypes.byref(p), 1)
    B, H, N, d = 2, 3, 256, 64
    assert fwd == 256
    assert bwd >= 256 + B * H * N * 4 + B * H * N * d * 4
    fake = ctypes.c_void_p(0x1000)
    assert lib.attn_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, None, 0, None) == \
        abi.ATTN_ERR_WORKSPACE
    assert lib.attn_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, ctypes.c_void_p(0x1010),
                        4096, None) == abi.ATTN_ERR_WORKSPACE          # misaligned
    assert lib.attn_bwd(ctypes.byref(p), *([fake] * 10), bwd - 1, None) == abi.ATTN_ERR_WORKSPACE
    # block masks add the compacted lists
    p2 = _params(abi, block_mask=0x2000, block_mask_head_stride=4)
    assert lib.attn_workspace_size(ctypes.byref(p2), 0) > fwd


def test_misaligned_tensor_is_rejected(abi):
    lib = abi.lib()
    p = _params(abi)
    ok = ctypes.c_void_p(0x1000)
    bad = ctypes.c_void_p(0x1008)
    st = lib.attn_fwd(ctypes.byref(p), ok, bad, ok, ok, ok, ok, 1 << 24, None)
    assert st == abi.ATTN_ERR_INVALID_ARG


def test_empty_problem_is_a_no_op(abi):
    lib = abi.lib()
    for f in ("N", "B", "H"):
        p = _params(abi, **{f: 0})
        st = lib.attn_fwd(ctypes.byref(p), None, None, None, None, None, ctypes.c_void_p(0x1000),
                          256, None)
        assert st == abi.ATTN_OK, (f, lib.attn_last_error())


def test_status_strings(abi):
    lib = abi.lib()
    for s in range(6):
        assert lib.attn_status_string(s)
    assert lib.attn_status_string(99) == b"unknown status"


def _decode_params(abi, **kw):
    # 2 sequences, 8 query heads over 2 key/value heads, caches of 1000 keys
    p = _params(abi, B=2, H=8, N=1000, d=128, H_kv=2, causal=1, key_lens=0x3000,
                stride_b=8 * 128, stride_h=128, stride_n=128,
                kv_stride_b=2 * 1000 * 128, kv_stride_h=1000 * 128, kv_stride_n=128)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_decode_workspace_holds_the_split_partials(abi):
    # 4 (b, kv head) pairs x 1000 keys is far below any split target, so the
    # cache splits into 256-key chunks whatever the device: 4 chunks, each
    # leaving fp32 O (d) and L per query row
    lib = abi.lib()
    p = _decode_params(abi)

    def up(x):
        return (x + 255) // 256 * 256

    for n_q in (1, 4, 16):
        rows = 2 * 8 * n_q
        want = 256 + up(4 * rows * 128 * 4) + up(4 * rows * 4)
        assert lib.attn_decode_workspace_size(ctypes.byref(p), n_q) == want, n_q


@pytest.mark.parametrize("kw,n_q,status", [
    (dict(dropout_p=0.1), 1, 2), (dict(block_mask=0x2000), 1, 2), (dict(key_lens=None), 1, 1),
    (dict(), 0, 1), (dict(), 17, 2),            # (H / H_kv) * n_q = 68 > 64 rows
    (dict(dtype=1), 1, 2), (dict(d=96), 1, 2),
])
def test_decode_options_checked_on_the_host(abi, kw, n_q, status):
    lib = abi.lib()
    p = _decode_params(abi, **kw)
    assert lib.attn_decode_workspace_size(ctypes.byref(p), n_q) == 0
    fake = ctypes.c_void_p(0x1000)
    st = lib.attn_decode(ctypes.byref(p), n_q, fake, fake, fake, fake, fake, fake, 1 << 30, None)
    assert st == status, lib.attn_last_error()
    assert lib.attn_last_error()


def test_noalloc_backward_checks_on_the_host(abi):
    lib = abi.lib()
    fake = ctypes.c_void_p(0x1000)
    # invalid parameters: the ordinary backward's status and message
    p = _params(abi, d=96)
    assert lib.attn_bwd_noalloc(ctypes.byref(p), *([fake] * 10), None) == \
        abi.ATTN_ERR_UNSUPPORTED
    assert lib.attn_last_error()
    # a problem whose scratch (here the 64 MiB fp32 dQ accumulator alone)
    # exceeds the built-in 64 MiB is refused before anything is enqueued
    p = _params(abi, B=1, H=16, N=8192, d=128, stride_b=16 * 8192 * 128, stride_h=8192 * 128,
                stride_n=128)
    assert lib.attn_workspace_size(ctypes.byref(p), 1) > 64 * 2 ** 20
    assert lib.attn_bwd_noalloc(ctypes.byref(p), *([fake] * 10), None) == abi.ATTN_ERR_WORKSPACE
    assert b"built-in scratch" in lib.attn_last_error()


def test_debug_stall_is_checked_on_the_host(abi):
    # arming touches no device: unknown kernels are refused, NONE disarms
    lib = abi.lib()
    assert lib.attn_debug_stall(7, 20_000_000) == abi.ATTN_ERR_INVALID_ARG
    assert b"unknown stall" in lib.attn_last_error()
    assert lib.attn_debug_stall(abi.ATTN_STALL_FWD_SOFTMAX, 0) == abi.ATTN_OK
    assert lib.attn_debug_stall(abi.ATTN_STALL_NONE, 0) == abi.ATTN_OK


def test_forward_splits_pairs_only_for_few_long_heads(abi):
    # pieces keep at least 8 key tiles: one head of N = 4096 (16 pairs of
    # 32 key tiles) is cut along the keys into 4 pieces; 16 heads x 64 pairs at
    # N = 16384 fill any GPU, and short rows are never cut
    lib = abi.lib()

    def ws(**kw):
        N = kw.get("N", 256)
        d = kw.get("d", 64)
        H = kw.get("H", 3)
        p = _params(abi, stride_b=H * N * d, stride_h=N * d, stride_n=d, **kw)
        return lib.attn_workspace_size(ctypes.byref(p), 0)

    assert ws(B=1, H=16, N=16384, d=128) == 256
    assert ws(B=2, H=3, N=1000) == 256
    # 128 pairs of 16 key tiles: more than half of any GPU's SMs, rows too
    # short to be worth the merge
    assert ws(B=1, H=16, N=2048, d=128) == 256
    nb, pieces = 32, 4
    rows = pieces * 1 * 1 * (nb // 2) * 256
    assert ws(B=1, H=1, N=4096, d=128) == 256 + rows * 128 * 4 + rows * 4
    # key padding without the causal mask keeps its longest-first order unsplit
    assert ws(B=1, H=1, N=4096, d=128, key_lens=0x3000) == 256
    assert ws(B=1, H=1, N=4096, d=128, key_lens=0x3000, causal=1) > 256


def test_backward_splits_key_tiles_only_for_few_long_heads(abi):
    # one head of 4096 keys has 32 key tiles for any GPU's SMs: each key
    # tile's 32 query tiles are cut into 4 pieces of 8, and the pieces' dK,
    # dV partials (fp32, [pieces][B*H_kv][nb*128][d] each) join the workspace
    lib = abi.lib()

    def ws(**kw):
        N, d, H = kw.get("N", 256), kw.get("d", 64), kw.get("H", 3)
        p = _params(abi, stride_b=H * N * d, stride_h=N * d, stride_n=d, **kw)
        return lib.attn_workspace_size(ctypes.byref(p), 1)

    N, d, nb = 4096, 128, 32
    base = 256 + 2 * N * 4 + N * d * 4          # row statistics + fp32 dQ accumulator
    assert ws(B=1, H=1, N=N, d=d) == base + 2 * 4 * nb * 128 * d * 4
    assert ws(B=1, H=16, N=16384, d=128) == 256 + 2 * 16 * 16384 * 4 + 16 * 16384 * 128 * 4
    assert ws(B=2, H=3, N=700) == 256 + 2 * 6 * 768 * 4 + 6 * 700 * 64 * 4   # short: unsplit
