"""The C-ABI library builds, loads and exports every symbol include/zq4.h
declares; host-side argument checks reject bad calls before any launch.
CPU only: no call here reaches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "zq4.h")).read()
    return sorted(set(re.findall(r"ZQ4_API\s+[\w\s\*]*?\b(zq4_\w+)\s*\(", text)))


def _cuda_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# The host-check tests pass fake device addresses that only the host checks
# look at. They run where no GPU can be reached, so that a broken check could
# never turn into a launch on those addresses.
host_checks_only = pytest.mark.skipif(_cuda_visible(), reason="fake device addresses: run without a GPU")


@pytest.fixture(scope="module")
def lib():
    from int4_weight_only_q4f16_gb300 import build
    build.build()
    from int4_weight_only_q4f16_gb300 import zq4
    return zq4


def test_header_declares_the_api():
    syms = declared_symbols()
    for s in ("zq4_gemv", "zq4_gate_up_silu", "zq4_moe_gemv", "zq4_prepare_weight",
              "zq4_dequant_f32", "zq4_dequant_f16", "zq4_status_string"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._build.LIB)
    for s in declared_symbols():
        assert hasattr(raw, s), s
    assert set(lib.EXPORTS) == set(declared_symbols())


def test_status_strings(lib):
    assert lib.status_string(0) == "ZQ4_OK"
    for st in range(-7, 0):
        assert lib.status_string(st).startswith("ZQ4_ERR")
    assert "unknown" in lib.status_string(-99)
    assert lib.lib.zq4_version() >= 100


def _call_gemv(lib, wq, sc, x, y, M, N, K):
    P = ctypes.c_void_p
    return lib.lib.zq4_gemv(P(wq), P(sc), P(x), P(y), M, N, K, P(0))


@host_checks_only
def test_host_checks_reject_before_launch(lib):
    A = 0x7F0000000000          # fake, 16-byte aligned, never dereferenced
    B, X, Y = A + (1 << 30), A + (2 << 30), A + (3 << 30)
    assert _call_gemv(lib, 0, B, X, Y, 1, 64, 64) == lib.ZQ4_ERR_NULL
    assert _call_gemv(lib, A, B, X, 0, 1, 64, 64) == lib.ZQ4_ERR_NULL
    assert _call_gemv(lib, A, B, X, Y, 1, 64, 48) == lib.ZQ4_ERR_SHAPE
    assert _call_gemv(lib, A, B, X, Y, 0, 64, 64) == lib.ZQ4_ERR_SHAPE
    assert _call_gemv(lib, A, B, X, Y, 1, 0, 64) == lib.ZQ4_ERR_SHAPE
    assert _call_gemv(lib, A + 4, B, X, Y, 1, 64, 64) == lib.ZQ4_ERR_ALIGN
    assert _call_gemv(lib, A, B, X + 2, Y, 1, 64, 64) == lib.ZQ4_ERR_ALIGN
    assert _call_gemv(lib, A, B, X, X, 1, 64, 64) == lib.ZQ4_ERR_OVERLAP
    assert _call_gemv(lib, A, B, X, A + 100, 1, 64, 64) == lib.ZQ4_ERR_OVERLAP
    P = ctypes.c_void_p
    # gate_up needs an even row count
    assert lib.lib.zq4_gate_up_silu(P(A), P(B), P(X), P(Y), 1, 63, 64, P(0)) == lib.ZQ4_ERR_SHAPE
    # MoE: unknown mode, missing router weights, top_k range
    ids, r = A + (4 << 30), A + (5 << 30)
    moe = lib.lib.zq4_moe_gemv
    assert moe(P(A), P(B), 4, P(X), P(Y), 1, 64, 64, P(ids), P(r), 2, 9, P(0), P(0)) == lib.ZQ4_ERR_FLAGS
    assert moe(P(A), P(B), 4, P(X), P(Y), 1, 64, 64, P(ids), P(0), 2, lib.MOE_DOWN_COMBINE,
               P(0), P(0)) == lib.ZQ4_ERR_NULL
    assert moe(P(A), P(B), 4, P(X), P(Y), 1, 64, 64, P(ids), P(r), 33, lib.MOE_DOWN_COMBINE,
               P(0), P(0)) == lib.ZQ4_ERR_SHAPE
    assert moe(P(A), P(B), 0, P(X), P(Y), 1, 64, 64, P(ids), P(r), 2, lib.MOE_DOWN_COMBINE,
               P(0), P(0)) == lib.ZQ4_ERR_SHAPE
    # prepare: odd N for interleave, unknown flag, overlap
    prep = lib.lib.zq4_prepare_weight
    assert prep(P(A), P(B), P(X), P(Y), 63, 64, 1, P(0)) == lib.ZQ4_ERR_SHAPE
    assert prep(P(A), P(B), P(X), P(Y), 64, 64, 7, P(0)) == lib.ZQ4_ERR_FLAGS
    assert prep(P(A), P(B), P(A), P(Y), 64, 64, 1, P(0)) == lib.ZQ4_ERR_OVERLAP
    # dequant
    assert lib.lib.zq4_dequant_f32(P(A), P(B), P(0), 4, 64, P(0)) == lib.ZQ4_ERR_NULL
    assert lib.lib.zq4_dequant_f16(P(A), P(B), P(Y), 4, 40, P(0)) == lib.ZQ4_ERR_SHAPE
    assert lib.lib.zq4_device_errors(P(0), 1) == lib.ZQ4_ERR_NULL


@host_checks_only
def test_affine_host_checks_reject_before_launch(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000          # fake, 16-byte aligned, never dereferenced
    S, Bi, X, Y = A + (1 << 30), A + (2 << 30), A + (3 << 30), A + (4 << 30)
    g = lib.lib.zq4_gemv_affine
    assert g(P(A), P(S), P(0), P(X), P(Y), 1, 64, 64, P(0)) == lib.ZQ4_ERR_NULL       # biases required
    assert g(P(A), P(S), P(Bi), P(X), P(Y), 1, 64, 96, P(0)) == lib.ZQ4_ERR_SHAPE     # K % 64
    assert g(P(A), P(S), P(Bi), P(X), P(Y), 0, 64, 64, P(0)) == lib.ZQ4_ERR_SHAPE
    assert g(P(A + 4), P(S), P(Bi), P(X), P(Y), 1, 64, 64, P(0)) == lib.ZQ4_ERR_ALIGN
    assert g(P(A), P(S + 1), P(Bi), P(X), P(Y), 1, 64, 64, P(0)) == lib.ZQ4_ERR_ALIGN
    assert g(P(A), P(S), P(Bi), P(X), P(Bi + 64), 1, 64, 64, P(0)) == lib.ZQ4_ERR_OVERLAP
    assert g(P(A), P(S), P(Bi), P(X), P(Y), 1, 64, 1 << 20, P(0)) == lib.ZQ4_ERR_UNSUPPORTED
    gu = lib.lib.zq4_gate_up_silu_affine
    assert gu(P(A), P(S), P(Bi), P(X), P(Y), 1, 63, 64, P(0)) == lib.ZQ4_ERR_SHAPE
    assert gu(P(A), P(S), P(Bi), P(X), P(X), 1, 64, 64, P(0)) == lib.ZQ4_ERR_OVERLAP


@host_checks_only
def test_affine_moe_host_checks(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000
    S, Bi, X, Y, ids, r = (A + (i << 30) for i in range(1, 7))
    m = lib.lib.zq4_moe_gemv_affine
    assert m(P(A), P(S), P(0), 4, P(X), P(Y), 1, 64, 64, P(ids), P(r), 2, lib.MOE_DOWN_COMBINE,
             P(0), P(0)) == lib.ZQ4_ERR_NULL
    assert m(P(A), P(S), P(Bi), 4, P(X), P(Y), 1, 64, 96, P(ids), P(r), 2, lib.MOE_DOWN_COMBINE,
             P(0), P(0)) == lib.ZQ4_ERR_SHAPE
    assert m(P(A), P(S), P(Bi), 4, P(X), P(Y), 1, 64, 64, P(ids), P(r), 2, 9, P(0), P(0)) == lib.ZQ4_ERR_FLAGS
    assert m(P(A), P(S + 1), P(Bi), 4, P(X), P(Y), 1, 64, 64, P(ids), P(r), 2, lib.MOE_DOWN_COMBINE,
             P(0), P(0)) == lib.ZQ4_ERR_ALIGN
    assert m(P(A), P(S), P(Bi), 4, P(X), P(Bi), 1, 64, 64, P(ids), P(r), 2, lib.MOE_DOWN_COMBINE,
             P(0), P(0)) == lib.ZQ4_ERR_OVERLAP


@host_checks_only
def test_add_rmsnorm_host_checks(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000
    S, X, R, G, O1, O2, W = (A + (i << 30) for i in range(1, 8))
    f = lib.lib.zq4_gemv_add_rmsnorm
    ok = (P(A), P(S), P(X), P(R), P(G), 1e-5, P(O1), P(O2), P(W), 1, 64, 64, P(0))
    assert lib.lib.zq4_add_rmsnorm_work_bytes(2, 64) == 16 + 2 * 64 * 4 + 4 * 64
    assert lib.lib.zq4_add_rmsnorm_work_bytes(0, 64) == 0
    args = list(ok); args[8] = P(0)
    assert f(*args) == lib.ZQ4_ERR_NULL
    args = list(ok); args[5] = -1.0
    assert f(*args) == lib.ZQ4_ERR_SHAPE                          # eps < 0
    args = list(ok); args[5] = float("nan")
    assert f(*args) == lib.ZQ4_ERR_SHAPE
    args = list(ok); args[8] = P(W + 8)
    assert f(*args) == lib.ZQ4_ERR_ALIGN                          # work 16-byte aligned
    args = list(ok); args[7] = P(O1 + 2)
    assert f(*args) == lib.ZQ4_ERR_OVERLAP                        # the two outputs
    args = list(ok); args[6] = P(R)
    assert f(*args) == lib.ZQ4_ERR_OVERLAP                        # res_out over resid (not in place)


@host_checks_only
def test_qkv_rope_host_checks(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000
    S, X, Pp, Sl, Q, Kc, Vc = (A + (i << 30) for i in range(1, 8))
    f = lib.lib.zq4_qkv_rope_append
    ok = [P(A), P(S), P(X), 1, 64, 4, 2, 8, 10000.0, P(Pp), P(Sl), P(Q), P(Kc), P(Vc), 16, P(0), P(0)]
    args = list(ok); args[7] = 7
    assert f(*args) == lib.ZQ4_ERR_SHAPE          # odd head dim
    args = list(ok); args[8] = 0.0
    assert f(*args) == lib.ZQ4_ERR_SHAPE          # rope base
    args = list(ok); args[9] = P(0)
    assert f(*args) == lib.ZQ4_ERR_NULL
    args = list(ok); args[10] = P(Sl + 2)
    assert f(*args) == lib.ZQ4_ERR_ALIGN
    args = list(ok); args[13] = P(Kc)
    assert f(*args) == lib.ZQ4_ERR_OVERLAP        # k and v caches the same


def test_moe_block_work_bytes_follow_the_documented_layout(lib):
    """The header's layout: 3 P + 3 int32 of grouping padded to 256 bytes,
    h [P, I] f16 padded to 256 bytes, z [P, D] fp32 (P = T top_k)."""
    def pad(n):
        return (n + 255) // 256 * 256
    for T, top_k, D, I in ((1, 8, 2048, 512), (16, 8, 2048, 512), (3, 5, 256, 768), (32, 8, 4096, 1536)):
        P = T * top_k
        assert lib.moe_block_work_bytes(T, top_k, D, I) == pad(4 * (3 * P + 3)) + pad(2 * P * I) + 4 * P * D
    for bad in ((0, 8, 256, 256), (1, 0, 256, 256), (1, 8, 0, 256), (1, 8, 256, -1)):
        assert lib.moe_block_work_bytes(*bad) == 0


@host_checks_only
def test_moe_block_host_checks(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000
    Dn, X, Y, ids, r, W = (A + (i << 30) for i in range(1, 7))
    T, top_k, D, I = 2, 8, 256, 512
    wb = lib.moe_block_work_bytes(T, top_k, D, I)
    f = lib.lib.zq4_moe_block
    ok = [P(A), P(Dn), 16, P(X), P(Y), T, D, I, P(ids), P(r), top_k, P(W), wb, P(0), P(0)]

    def call(**change):
        args = list(ok)
        for i, v in change.items():
            args[int(i[1:])] = v
        return f(*args)
    for i in (0, 1, 3, 4, 8, 9, 11):
        assert call(**{f"a{i}": P(0)}) == lib.ZQ4_ERR_NULL, i
    assert call(a2=0) == lib.ZQ4_ERR_SHAPE                       # no experts
    assert call(a5=0) == lib.ZQ4_ERR_SHAPE                       # no tokens
    assert call(a10=33) == lib.ZQ4_ERR_SHAPE                     # top_k above 32
    assert call(a6=320) == lib.ZQ4_ERR_SHAPE                     # D not a multiple of 256
    assert call(a7=192) == lib.ZQ4_ERR_SHAPE                     # I not a multiple of 256
    assert call(a5=33) == lib.ZQ4_ERR_UNSUPPORTED                # 264 pairs
    assert call(a12=wb - 1) == lib.ZQ4_ERR_SHAPE                 # scratch too small
    assert call(a0=P(A + 4)) == lib.ZQ4_ERR_ALIGN
    assert call(a11=P(W + 8)) == lib.ZQ4_ERR_ALIGN               # work 16-byte aligned
    assert call(a8=P(ids + 2)) == lib.ZQ4_ERR_ALIGN
    assert call(a4=P(X + 32)) == lib.ZQ4_ERR_OVERLAP             # y over x
    assert call(a11=P(r)) == lib.ZQ4_ERR_OVERLAP                 # work over the router weights


def test_header_is_plain_c_and_a_c_program_links(lib):
    """include/zq4.h compiles as strict C99 (no C++ in the boundary), every
    declared entry point resolves when a C program links libzq4.so, and the
    host checks answer a C caller (a NULL matrix: ZQ4_ERR_NULL, no launch)."""
    import shutil
    import subprocess
    from int4_weight_only_q4f16_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    syms = declared_symbols()
    out_dir = os.path.join(build.BUILD, "c_abi_check")
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "c_abi_check.c")
    exe = os.path.join(out_dir, "c_abi_check")
    table = ",\n".join(f"    (zq4_fn){s}" for s in syms)
    with open(src, "w") as f:
        f.write(f"""#include <stdio.h>
#include "zq4.h"

typedef void (*zq4_fn)(void);
static zq4_fn const every_entry[] = {{
{table}
}};

int main(void)
{{
    size_t i, n = sizeof every_entry / sizeof every_entry[0];
    int bad = 0;
    for (i = 0; i < n; ++i)
        if (!every_entry[i]) ++bad;
    if (zq4_version() <= 0) ++bad;
    if (zq4_gemv(NULL, NULL, NULL, NULL, 1, 64, 64, NULL) != ZQ4_ERR_NULL) ++bad;
    if (!zq4_status_string(ZQ4_ERR_SHAPE)) ++bad;
    printf("%lu %d\\n", (unsigned long)n, bad);
    return bad;
}}
""")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           src, "-o", exe, "-L", build.BUILD, "-lzq4", f"-Wl,-rpath,{build.BUILD}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == [str(len(syms)), "0"]


def test_binding_structs_match_the_header_layout(lib):
    """The binding's ctypes mirrors of zq4_stack_job and zq4_stack_plan have
    the C compiler's size and field offsets for include/zq4.h."""
    import ctypes
    import shutil
    import subprocess
    from int4_weight_only_q4f16_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mirrors = {"zq4_stack_job": lib.StackJob, "zq4_stack_plan": lib.StackPlanC}
    lines = []
    for cname, py in mirrors.items():
        lines.append(f'    printf("{cname} size %lu\\n", (unsigned long)sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'    printf("{cname} {field} %lu\\n", (unsigned long)offsetof({cname}, {field}));')
    out_dir = os.path.join(build.BUILD, "c_abi_check")
    os.makedirs(out_dir, exist_ok=True)
    src, exe = os.path.join(out_dir, "c_layout.c"), os.path.join(out_dir, "c_layout")
    with open(src, "w") as f:
        f.write("#include <stddef.h>\n#include <stdio.h>\n#include \"zq4.h\"\n\nint main(void)\n{\n" +
                "\n".join(lines) + "\n    return 0;\n}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0
    got = {}
    for line in r.stdout.split("\n"):
        if line:
            cname, field, v = line.split()
            got[(cname, field)] = int(v)
    for cname, py in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert got[(cname, field)] == getattr(py, field).offset, (cname, field)


def test_host_only_calls(lib):
    """Calls that never touch a device: the segmented layout's size (one
    2304-byte segment per 16-row tile and 256-column block) and the plan's
    wait limit (0 restores the 2 s default)."""
    import ctypes
    sb = lib.lib.zq4_segmented_bytes
    for N, K in ((1, 256), (16, 256), (17, 512), (3072, 3072), (32064, 3072)):
        assert sb(N, K) == (N + 15) // 16 * (K // 256) * 2304, (N, K)
    for N, K in ((0, 256), (16, 128), (16, 0), (-1, 256)):
        assert sb(N, K) == 0, (N, K)
    plan = lib.StackPlanC()
    f = lib.lib.zq4_stack_plan_set_wait_limit
    assert f(None, 5) == lib.ZQ4_ERR_NULL
    assert f(ctypes.byref(plan), 5_000_000) == lib.ZQ4_OK and plan.wait_ns == 5_000_000
    assert f(ctypes.byref(plan), 0) == lib.ZQ4_OK and plan.wait_ns == 2_000_000_000
    nbytes = ctypes.c_size_t(0)
    job = lib.StackJob()
    assert lib.lib.zq4_stack_plan_bytes(ctypes.byref(job), 1, 1, None) == lib.ZQ4_ERR_NULL
    assert lib.lib.zq4_stack_plan_bytes(None, 1, 1, ctypes.byref(nbytes)) == lib.ZQ4_ERR_NULL
    assert lib.lib.zq4_stack_plan_bytes(ctypes.byref(job), 0, 1, ctypes.byref(nbytes)) == lib.ZQ4_ERR_SHAPE


@host_checks_only
def test_argmax_and_segmented_host_checks(lib):
    P = ctypes.c_void_p
    A = 0x7F0000000000
    S, X, Y32, Ix, Mx, W = (A + (i << 30) for i in range(1, 7))
    am = lib.lib.zq4_gemv_argmax
    ok = [P(A), P(S), P(X), P(Y32), P(Ix), P(Mx), P(W), 1, 64, 256, P(0)]

    def call(f, base, **change):
        args = list(base)
        for i, v in change.items():
            args[int(i[1:])] = v
        return f(*args)
    for i in (2, 4, 6):
        assert call(am, ok, **{f"a{i}": P(0)}) == lib.ZQ4_ERR_NULL, i
    assert call(am, ok, a7=0) == lib.ZQ4_ERR_SHAPE
    assert call(am, ok, a7=65) == lib.ZQ4_ERR_SHAPE              # at most 64 tokens
    assert call(am, ok, a2=P(X + 2)) == lib.ZQ4_ERR_ALIGN
    assert call(am, ok, a4=P(Ix + 2)) == lib.ZQ4_ERR_ALIGN
    assert call(am, ok, a6=P(W + 4)) == lib.ZQ4_ERR_ALIGN          # keys 8-byte aligned
    for f, gate_up in ((lib.lib.zq4_gemv_seg, False), (lib.lib.zq4_gate_up_silu_seg, True)):
        base = [P(A), P(X), P(Y32), 1, 64, 256, P(0)]
        assert call(f, base, a0=P(0)) == lib.ZQ4_ERR_NULL
        assert call(f, base, a2=P(0)) == lib.ZQ4_ERR_NULL
        assert call(f, base, a5=128) == lib.ZQ4_ERR_SHAPE          # K % 256
        assert call(f, base, a3=0) == lib.ZQ4_ERR_SHAPE
        assert call(f, base, a0=P(A + 4)) == lib.ZQ4_ERR_ALIGN
        assert call(f, base, a1=P(X + 2)) == lib.ZQ4_ERR_ALIGN
        assert call(f, base, a2=P(Y32 + 1)) == lib.ZQ4_ERR_ALIGN
        if gate_up:
            assert call(f, base, a4=63) == lib.ZQ4_ERR_SHAPE


def test_binding_fails_loudly_without_the_library():
    """No CPU fallback: with libzq4.so absent, importing the binding (and the
    decode-stack driver that uses it) raises ImportError."""
    import subprocess
    import sys
    code = (
        "import os\n"
        "import int4_weight_only_q4f16_gb300.build as b\n"
        "b.LIB = os.path.join(b.BUILD, 'absent', 'libzq4.so')\n"
        "for mod in ('zq4', 'stack'):\n"
        "    try:\n"
        "        __import__('int4_weight_only_q4f16_gb300.' + mod)\n"
        "    except ImportError as e:\n"
        "        print(mod, 'ImportError', 'not built' in str(e))\n"
        "    else:\n"
        "        print(mod, 'loaded')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split("\n")[:2] == ["zq4 ImportError True", "stack ImportError True"], r.stdout
