"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every
function include/attn.h declares, and its host-side argument checks return the
documented codes before touching CUDA."""

import ctypes
import os
import re
import subprocess
import sys

import pytest

from exact_attention_86_gb300 import attn
from exact_attention_86_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return attn.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(attn_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert {"attn_fwd", "attn_get_error_string", "attn_check_device_status",
            "attn_selftest_wait_timeout", "attn_abi_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) <= set(attn.SIGNATURES)


def test_abi_version(lib):
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    ver = int(re.search(r"#define ATTN_ABI_VERSION (\d+)", src).group(1))
    assert attn.attn_abi_version() == ver


def test_error_strings(lib):
    for code in range(10):
        assert attn.attn_get_error_string(code) not in ("", "unknown status")
    assert attn.attn_get_error_string(99) == "unknown status"


A = 1 << 20  # a 16-byte-aligned dummy address: argument checks never dereference


@pytest.mark.parametrize("args,code", [
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(B=-1), attn.ATTN_ERR_SHAPE),
    (dict(Sq=-5), attn.ATTN_ERR_SHAPE),
    (dict(Sk=-1), attn.ATTN_ERR_SHAPE),
    (dict(scale=float("nan")), attn.ATTN_ERR_SCALE),
    (dict(scale=float("inf")), attn.ATTN_ERR_SCALE),
    (dict(q=0), attn.ATTN_ERR_NULLPTR),
    (dict(o=0), attn.ATTN_ERR_NULLPTR),
    (dict(lse=0), attn.ATTN_ERR_NULLPTR),
    (dict(k=0), attn.ATTN_ERR_NULLPTR),
    (dict(q=A + 8), attn.ATTN_ERR_ALIGN),
    (dict(v=A + 2), attn.ATTN_ERR_ALIGN),
    (dict(lse=A + 2), attn.ATTN_ERR_ALIGN),
    (dict(kv=A + 1), attn.ATTN_ERR_ALIGN),
    (dict(H=1 << 20, Sq=1 << 20, Sk=1 << 20), attn.ATTN_ERR_SHAPE),
    (dict(B=0), attn.ATTN_OK),      # nothing to compute, no launch
    (dict(Sq=0), attn.ATTN_OK),
    (dict(H=0, q=0, o=0), attn.ATTN_OK),
])
def test_argument_checks(lib, args, code):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=2, H=2, Sq=256, Sk=256, D=128, scale=0.088, causal=0, kv=None)
    a.update(args)
    st = attn.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Sq"], a["Sk"], a["D"],
                       a["scale"], a["causal"], a["kv"], None)
    assert st == code


def test_no_silent_success_without_gpu(lib):
    # The calls run in a child process that sees no device at all
    # (CUDA_VISIBLE_DEVICES empty), so whatever machine runs this test, the
    # shapes below, which pass every host-side check, can never reach a launch
    # with the dummy addresses: the library must report an error instead of
    # success.
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from exact_attention_86_gb300 import attn\n"
        "A = 1 << 20\n"
        "st = attn.attn_fwd(A, A, A, A, A, 1, 1, 128, 128, 64, 0.125, 0, None, None)\n"
        "sf = attn.attn_selftest_wait_timeout(1000, None)\n"
        "print(st, sf)\n" % ROOT)
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    st, sf = (int(x) for x in out.stdout.split())
    assert st in (attn.ATTN_ERR_CUDA, attn.ATTN_ERR_UNSUPPORTED_DEVICE)
    assert sf in (attn.ATTN_ERR_CUDA, attn.ATTN_ERR_UNSUPPORTED_DEVICE)


def test_selftest_limit_checked(lib):
    assert attn.attn_selftest_wait_timeout(0, None) == attn.ATTN_ERR_SHAPE
    assert attn.attn_selftest_wait_timeout(3_000_000_000, None) == attn.ATTN_ERR_SHAPE


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "exact_attention_86_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", src, flags=re.M), fn
                assert "oracle/" not in src, fn


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(attn, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(attn, "_lib", None)
    with pytest.raises(RuntimeError):
        attn.lib()


W = 1 << 24  # a 256-byte-aligned dummy workspace address


@pytest.mark.parametrize("args,code", [
    (dict(ns=0), attn.ATTN_ERR_SHAPE),
    (dict(ns=129), attn.ATTN_ERR_SHAPE),
    (dict(ws=0), attn.ATTN_ERR_NULLPTR),
    (dict(ws=W + 128), attn.ATTN_ERR_ALIGN),
    (dict(wsb=1024), attn.ATTN_ERR_WORKSPACE),
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(Sq=0), attn.ATTN_OK),
])
def test_splitkv_argument_checks(lib, args, code):
    a = dict(B=2, H=2, Sq=256, Sk=512, D=128, ns=4, ws=W, wsb=None)
    a.update(args)
    need = attn.attn_fwd_splitkv_workspace_size(a["B"], a["H"], a["Sq"], a["D"], a["ns"]) if a["D"] in (64, 128) else 0
    wsb = need if a["wsb"] is None else a["wsb"]
    st = attn.attn_fwd_splitkv(A, A, A, A, A, a["B"], a["H"], a["Sq"], a["Sk"], a["D"], 0.1, 0, None, a["ns"],
                               a["ws"], wsb, None)
    assert st == code


def test_splitkv_workspace_size(lib):
    # fp32 partial O and LSE for every split, each part rounded up to 256 bytes
    rows = 2 * 3 * 300
    o_bytes = -(-(5 * rows * 128 * 4) // 256) * 256
    l_bytes = -(-(5 * rows * 4) // 256) * 256
    assert attn.attn_fwd_splitkv_workspace_size(2, 3, 300, 128, 5) == o_bytes + l_bytes
    assert attn.attn_fwd_splitkv_workspace_size(2, 3, 300, 96, 5) == 0
    assert attn.attn_fwd_splitkv_workspace_size(2, 3, 300, 128, 0) == 0


@pytest.mark.parametrize("args,code", [
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(n=0), attn.ATTN_ERR_SHAPE),
    (dict(rows=-1), attn.ATTN_ERR_SHAPE),
    (dict(op=0), attn.ATTN_ERR_NULLPTR),
    (dict(op=A + 4), attn.ATTN_ERR_ALIGN),
    (dict(rows=0), attn.ATTN_OK),
])
def test_merge_argument_checks(lib, args, code):
    a = dict(op=A, lp=A, n=3, o=A, lse=A, rows=100, D=128)
    a.update(args)
    assert attn.attn_lse_merge(a["op"], a["lp"], a["n"], a["o"], a["lse"], a["rows"], a["D"], None) == code


@pytest.mark.parametrize("args,code", [
    (dict(D=100), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(batch=-1), attn.ATTN_ERR_SHAPE),
    (dict(tq=-1), attn.ATTN_ERR_SHAPE),
    (dict(cq=0), attn.ATTN_ERR_NULLPTR),
    (dict(ck=0), attn.ATTN_ERR_NULLPTR),
    (dict(cq=A + 2), attn.ATTN_ERR_ALIGN),
    (dict(q=A + 8), attn.ATTN_ERR_ALIGN),
    (dict(scale=float("nan")), attn.ATTN_ERR_SCALE),
    (dict(batch=0), attn.ATTN_OK),
    (dict(tq=0), attn.ATTN_OK),
    (dict(maxq=0), attn.ATTN_OK),
    (dict(tc=A + 4), attn.ATTN_ERR_ALIGN),
])
def test_varlen_argument_checks(lib, args, code):
    a = dict(q=A, k=A, v=A, o=A, lse=A, cq=A, ck=A, batch=3, maxq=300, tq=600, tk=700, H=4, D=128, scale=0.1,
             tc=None)
    a.update(args)
    st = attn.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], a["batch"], a["maxq"],
                              a["tq"], a["tk"], a["H"], a["D"], a["scale"], 0, a["tc"], None)
    assert st == code


@pytest.mark.parametrize("args,code", [
    (dict(D=100), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(ps=96), attn.ATTN_ERR_SHAPE),
    (dict(ps=32), attn.ATTN_ERR_SHAPE),
    (dict(npg=0), attn.ATTN_ERR_SHAPE),
    (dict(mp=0), attn.ATTN_ERR_SHAPE),
    (dict(npg=1 << 30), attn.ATTN_ERR_SHAPE),
    (dict(bt=0), attn.ATTN_ERR_NULLPTR),
    (dict(sk=0), attn.ATTN_ERR_NULLPTR),
    (dict(kc=A + 8), attn.ATTN_ERR_ALIGN),
    (dict(bt=A + 2), attn.ATTN_ERR_ALIGN),
    (dict(scale=float("inf")), attn.ATTN_ERR_SCALE),
    (dict(batch=0), attn.ATTN_OK),
    (dict(tq=0), attn.ATTN_OK),
    (dict(tc=A + 4), attn.ATTN_ERR_ALIGN),
])
def test_paged_argument_checks(lib, args, code):
    # every case ends in a host-side check (no launch, with or without a GPU)
    a = dict(q=A, kc=A, vc=A, o=A, lse=A, cq=A, sk=A, bt=A, batch=3, maxq=300, tq=600, npg=40, ps=128, mp=8, H=4,
             D=128, scale=0.1, tc=None)
    a.update(args)
    st = attn.attn_fwd_paged(a["q"], a["kc"], a["vc"], a["o"], a["lse"], a["cq"], a["sk"], a["bt"], a["batch"],
                             a["maxq"], a["tq"], a["npg"], a["ps"], a["mp"], a["H"], a["D"], a["scale"], 0, a["tc"],
                             None)
    assert st == code


@pytest.mark.parametrize("args,code", [
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(Sk=200), attn.ATTN_ERR_SHAPE),
    (dict(B=-1), attn.ATTN_ERR_SHAPE),
    (dict(scale=float("nan")), attn.ATTN_ERR_SCALE),
    (dict(qd=float("inf")), attn.ATTN_ERR_SCALE),
    (dict(vd=float("nan")), attn.ATTN_ERR_SCALE),
    (dict(qd=3e38, kd=3e38), attn.ATTN_ERR_SCALE),
    (dict(q=0), attn.ATTN_ERR_NULLPTR),
    (dict(v=0), attn.ATTN_ERR_NULLPTR),
    (dict(v=A + 8), attn.ATTN_ERR_ALIGN),
    (dict(kv=A + 2), attn.ATTN_ERR_ALIGN),
    (dict(B=0), attn.ATTN_OK),
    (dict(Sq=0), attn.ATTN_OK),
])
def test_fp8_argument_checks(lib, args, code):
    # every case ends in a host-side check (no launch, with or without a GPU)
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=2, H=2, Sq=256, Sk=256, D=128, scale=0.088, kv=None, qd=1.0, kd=1.0,
             vd=1.0)
    a.update(args)
    st = attn.attn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Sq"], a["Sk"], a["D"],
                           a["scale"], 0, a["kv"], a["qd"], a["kd"], a["vd"], None)
    assert st == code


@pytest.mark.parametrize("args,code", [
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED_D),
    (dict(Sk=-1), attn.ATTN_ERR_SHAPE),
    (dict(scale=float("nan")), attn.ATTN_ERR_SCALE),
    (dict(dout=0), attn.ATTN_ERR_NULLPTR),
    (dict(dq=0), attn.ATTN_ERR_NULLPTR),
    (dict(dk=0), attn.ATTN_ERR_NULLPTR),
    (dict(ws=0), attn.ATTN_ERR_NULLPTR),
    (dict(dv=A + 8), attn.ATTN_ERR_ALIGN),
    (dict(ws=A + 64), attn.ATTN_ERR_ALIGN),
    (dict(wsb=16), attn.ATTN_ERR_WORKSPACE),
    (dict(B=0), attn.ATTN_OK),
    (dict(Sq=0, Sk=0), attn.ATTN_OK),
])
def test_bwd_argument_checks(lib, args, code):
    # every case ends in a host-side check (no launch, with or without a GPU)
    a = dict(dout=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 20, B=2, H=2, Sq=256, Sk=256, D=128, scale=0.1)
    a.update(args)
    st = attn.attn_bwd(A, A, A, A, a["dout"], A, a["dq"], a["dk"], a["dv"], a["B"], a["H"], a["Sq"], a["Sk"], a["D"],
                       a["scale"], 0, None, a["ws"], a["wsb"], None)
    assert st == code


def test_bwd_workspace_size(lib):
    assert attn.attn_bwd_workspace_size(2, 3, 300) == -(-(2 * 3 * 300 * 4) // 256) * 256
    assert attn.attn_bwd_workspace_size(-1, 3, 300) == 0


def test_launch_floor_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    assert attn.attn_selftest_launch_floor(0, 64, 0, None) == attn.ATTN_ERR_SHAPE
    assert attn.attn_selftest_launch_floor(70000, 64, 0, None) == attn.ATTN_ERR_SHAPE
    assert attn.attn_selftest_launch_floor(1, 64, 2, None) == attn.ATTN_ERR_SHAPE
    assert attn.attn_selftest_launch_floor(1, 96, 0, None) == attn.ATTN_ERR_UNSUPPORTED_D


def test_kernel_choice(lib):
    # host-only model of which padded-forward kernel runs (no device call);
    # arguments B, H, Sq, Sk, D, causal, num_sms
    f = attn.attn_fwd_kernel_choice
    assert f(2, 16, 8192, 8192, 128, 0, 152) == 1   # 1024 pairs: 7 waves against 14 of single tiles
    assert f(8, 16, 2048, 2048, 128, 0, 152) == 1
    assert f(2, 16, 8192, 8192, 128, 1, 152) == 1   # causal, 1024 pair units dealt statically
    assert f(1, 8, 32768, 32768, 128, 1, 152) == 1
    assert f(4, 8, 1024, 1024, 128, 1, 152) == 0    # causal, short: the longest pair unit sets the time
    assert f(2, 16, 2048, 2048, 128, 1, 152) == 0   # causal, 8 pairs a head: unit costs favour single tiles
    assert f(8, 16, 2048, 2048, 128, 1, 152) == 0   # (measured 148 against 154 us)
    assert f(2, 16, 4096, 4096, 128, 1, 152) == 1   # (measured 128 against 132 us)
    assert f(16, 16, 8192, 8192, 128, 1, 152) == 0  # causal, 8192 pair units: more than the static deal holds
    assert f(1, 8, 128, 32768, 128, 0, 152) == 0    # one query tile per head: pairs half empty
    assert f(1, 1, 128, 128, 128, 0, 152) == 0
    assert f(1, 1, 8192, 8192, 128, 0, 152) == 0    # 64 single tiles fit one wave
    assert f(0, 16, 8192, 8192, 128, 0, 152) == 0
    # D = 64: lighter products, so the pair more often (measured)
    assert f(8, 16, 1024, 1024, 64, 0, 152) == 1    # 4 against 7 waves (58 against 66 us)
    assert f(8, 16, 1024, 1024, 128, 0, 152) == 0   # the same waves at D = 128 favour single tiles
    assert f(8, 16, 2048, 2048, 64, 1, 152) == 1    # causal (130 against 138 us)
    assert f(8, 16, 1024, 1024, 64, 1, 152) == 0    # causal (52 against 50 us)
    assert f(-1, 16, 8192, 8192, 128, 0, 152) == -1
    assert f(2, 16, 8192, -1, 128, 0, 152) == -1
    assert f(2, 16, 8192, 8192, 128, 0, -1) == -1
    assert f(2, 16, 8192, 8192, 96, 0, 152) == -1   # unsupported D
    # never for a single query tile, whatever the batch
    for bh in (1, 7, 152, 153, 10_000):
        for causal in (0, 1):
            for D in (64, 128):
                assert f(1, bh, 100, 100, D, causal, 152) == 0
                assert f(1, bh, 128, 4096, D, causal, 152) == 0
    # E4M3: the two-tile kernel measured faster on every batch above one query tile timed
    f8 = attn.attn_fwd_fp8_kernel_choice
    assert f8(8, 16, 2048, 2048, 128, 1, 152) == 1  # causal (136 against 156 us)
    assert f8(8, 16, 1024, 1024, 128, 1, 152) == 1  # causal (54 against 56 us)
    assert f8(2, 16, 4096, 4096, 128, 0, 152) == 1  # non-causal, 4 against 7 waves (201 against 214 us)
    assert f8(2, 16, 8192, 8192, 128, 0, 152) == 1
    assert f8(1, 8, 128, 32768, 128, 0, 152) == 0   # one query tile per head
    assert f8(1, 1, 8192, 8192, 128, 0, 152) == 0   # 64 single tiles fit one wave
    assert f8(16, 16, 8192, 8192, 128, 1, 152) == 0  # more units than the static deal holds
    assert f8(-1, 16, 8192, 8192, 128, 0, 152) == -1


def test_fwd_abort_selftest_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    f = attn.attn_selftest_fwd_abort
    a = (A, A, A, A, A, 1, 2, 256)
    assert f(*a, 256, 128, 0.1, 0, None, -1, 0, 999, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 256, 128, 0.1, 0, None, -1, 0, 3_000_000_000, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 256, 128, 0.1, 0, None, -1, -1, 10_000, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 0, 128, 0.1, 0, None, -1, 0, 10_000, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 256, 96, 0.1, 0, None, -1, 0, 10_000, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(A + 8, *a[1:], 256, 128, 0.1, 0, None, -1, 0, 10_000, None) == attn.ATTN_ERR_ALIGN
    assert f(*a, 256, 128, 0.1, 0, None, 2, 0, 10_000, None) == attn.ATTN_ERR_SHAPE    # unknown kernel


def test_variant_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    f = attn.attn_fwd_variant
    a = (A, A, A, A, A, 1, 2, 256, 256)
    assert f(*a, 128, 0.1, 0, None, 2, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 128, 0.1, 0, None, -2, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 96, 0.1, 0, None, attn.ATTN_KERNEL_ONE_TILE, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(*a, 128, float("inf"), 0, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SCALE
    assert f(A, None, A, A, A, 1, 2, 256, 256, 128, 0.1, 0, None, -1, None) == attn.ATTN_ERR_NULLPTR
    # nothing to compute: OK without a device query or a launch
    assert f(*a[:5], 0, 2, 256, 256, 128, 0.1, 0, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_OK


def test_varlen_and_paged_variant_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    f = attn.attn_fwd_varlen_variant
    a = (A, A, A, A, A, A, A, 2, 256, 512, 512, 2)  # ... batch, max_seqlen_q, total_q, total_k, H
    assert f(*a, 128, 0.1, 1, None, 2, None) == attn.ATTN_ERR_SHAPE                     # unknown kernel
    assert f(*a, 128, 0.1, 1, None, -2, None) == attn.ATTN_ERR_SHAPE
    assert f(*a, 96, 0.1, 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(*a, 128, float("nan"), 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SCALE
    assert f(A, A, A, None, *a[4:], 128, 0.1, 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_NULLPTR
    assert f(A + 8, *a[1:], 128, 0.1, 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_ALIGN
    assert f(*a, 128, 0.1, 1, A + 4, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_ALIGN  # counter
    assert f(A, A, A, A, A, A, A, 0, 256, 512, 512, 2, 128, 0.1, 1, None,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_OK                                    # nothing to compute
    g = attn.attn_fwd_paged_variant
    b = (A, A, A, A, A, A, A, A, 2, 256, 512)  # ... block_table, batch, max_seqlen_q, total_q
    assert g(*b, 4, 256, 2, 2, 128, 0.1, 1, None, 2, None) == attn.ATTN_ERR_SHAPE       # unknown kernel
    assert g(*b, 4, 100, 2, 2, 128, 0.1, 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SHAPE
    assert g(*b, 0, 256, 2, 2, 128, 0.1, 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SHAPE
    assert g(*b, 4, 256, 2, 2, 96, 0.1, 1, None, attn.ATTN_KERNEL_ONE_TILE, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert g(*b, 4, 256, 2, 2, 128, float("inf"), 1, None, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SCALE
    assert g(*b[:7], None, *b[8:], 4, 256, 2, 2, 128, 0.1, 1, None,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_NULLPTR                           # no page table
    assert g(A, A + 8, *b[2:], 4, 256, 2, 2, 128, 0.1, 1, None,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_ALIGN
    assert g(*b[:8], 0, 256, 512, 4, 256, 2, 2, 128, 0.1, 1, None,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_OK                                    # nothing to compute


def test_fp8_ex_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    f = attn.attn_fwd_fp8_ex
    args = (A, A, A, A, A, 1, 2, 256, 256)
    assert f(*args, 128, 0.1, 0, None, 1.0, 1.0, 1.0, 2, None) == attn.ATTN_ERR_SHAPE      # unknown layout
    assert f(*args, 128, 0.1, 0, None, 1.0, 1.0, 1.0, -1, None) == attn.ATTN_ERR_SHAPE
    assert f(*args, 96, 0.1, 0, None, 1.0, 1.0, 1.0, 0, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(*args, 32, 0.1, 0, None, 1.0, 1.0, 1.0, 1, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(A, A, A, A, A, 1, 2, 256, 100, 128, 0.1, 0, None, 1.0, 1.0, 1.0, 1, None) == attn.ATTN_ERR_SHAPE
    assert f(*args, 128, float("nan"), 0, None, 1.0, 1.0, 1.0, 0, None) == attn.ATTN_ERR_SCALE
    assert f(A + 8, A, A, A, A, 1, 2, 256, 256, 128, 0.1, 0, None, 1.0, 1.0, 1.0, 0, None) == attn.ATTN_ERR_ALIGN


def test_fp8_variant_argument_checks(lib):
    # each call ends at a host-side check (no device query, no launch)
    f = attn.attn_fwd_fp8_variant
    args = (A, A, A, A, A, 1, 2, 256, 256, 128, 0.1, 0, None, 1.0, 1.0, 1.0)
    assert f(*args, attn.ATTN_V_ROWS, 2, None) == attn.ATTN_ERR_SHAPE                   # unknown kernel
    assert f(*args, attn.ATTN_V_ROWS, -2, None) == attn.ATTN_ERR_SHAPE
    assert f(*args, 5, attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_SHAPE         # unknown layout
    assert f(A, A, A, A, A, 1, 2, 256, 256, 96, 0.1, 0, None, 1.0, 1.0, 1.0, attn.ATTN_V_ROWS,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_ERR_UNSUPPORTED_D
    assert f(A, A, A, A, A, 0, 2, 256, 256, 128, 0.1, 0, None, 1.0, 1.0, 1.0, attn.ATTN_V_ROWS,
             attn.ATTN_KERNEL_TWO_TILE, None) == attn.ATTN_OK                             # nothing to compute
