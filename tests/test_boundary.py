"""Host-only checks of the C-ABI library: it loads, exports every symbol that
include/fa.h declares, and rejects invalid calls with the documented status
codes before touching the GPU (no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build_library()
    from attention_fa_fwd_02_gb300 import fa as fa_mod
    return fa_mod


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return set(re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text))


def test_header_declares_the_abi():
    assert _declared_symbols() == {"fa_fwd", "fa_bwd", "fa_device_status", "fa_status_string",
                                   "fa_version", "fa_timing_enable", "fa_timing_read",
                                   "fa_fwd_noalloc", "fa_selftest_timeout",
                                   "fa_noalloc_scratch_bytes", "fa_bwd_dsmat"}


def test_noalloc_scratch_size_matches_the_header(fa):
    # the binding reads the size from the library; it must be the header's value
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \(\(unsigned long long\)(\d+) << (\d+)\)", text)
    assert m, "FA_NOALLOC_SCRATCH_BYTES definition not found"
    assert fa.noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_library_exports_every_declared_symbol(fa):
    lib = fa.lib()
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {fa.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    assert _declared_symbols() <= exported
    # hidden visibility: nothing but the ABI leaks out of the library
    assert exported == _declared_symbols()


def test_timing_read_empty(fa):
    # nothing recorded: no CUDA call needed, zero kernels reported
    assert fa.fa_timing_enable(False) == 0
    assert fa.fa_timing_read() == {}


def test_selftest_timeout_rejects_bad_args(fa):
    assert fa.fa_selftest_timeout(1000, 0, 0) == 1          # null counter
    assert fa.fa_selftest_timeout(0, A, 0) == 1             # zero limit
    assert fa.fa_selftest_timeout(20 * 10**9, A, 0) == 1    # limit above 10 s
    assert fa.fa_selftest_timeout(1000, MIS, 0) == 3        # misaligned counter


def test_status_strings(fa):
    assert fa.status_string(0) == "ok"
    for code in range(1, 7):
        assert fa.status_string(code) and fa.status_string(code) != "unknown status"
    assert fa.status_string(99) == "unknown status"
    assert fa.version().startswith("fa-sm103a")


def _params(fa, **kw):
    d = dict(B=1, H=4, HKV=2, Sq=128, Sk=128, D=128, scale=0.088, causal=1, window=0,
             in_dtype=fa.FA_BF16, out_dtype=fa.FA_F32)
    d.update(kw)
    return fa.fa_params(**d)


# Fake, never-dereferenced addresses: every call below must be rejected by
# validation before any CUDA call is made.
A = 0x10000
MIS = 0x10008


@pytest.mark.parametrize("kw,code", [
    (dict(H=3, HKV=2), 1),          # H % HKV != 0
    (dict(B=0), 1),
    (dict(HKV=0), 1),
    (dict(Sq=-1), 1),
    (dict(D=0), 1),
    (dict(scale=0.0), 1),
    (dict(scale=-0.1), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(causal=2), 1),
    (dict(window=-1), 1),
    (dict(in_dtype=7), 1),
    (dict(out_dtype=-1), 1),
    (dict(D=24), 2),                # head dim not a multiple of 16
    (dict(D=144), 2),               # above 128
    (dict(D=8), 2),
    (dict(D=144, in_dtype=0), 2),   # fp32 inputs up to D=128 too
    (dict(D=40, in_dtype=0), 2),
    (dict(f32_mma=2), 1),           # not an fa_f32_mma value (checked for bf16 inputs too)
    (dict(f32_mma=-1, in_dtype=0), 1),
    (dict(D=80, in_dtype=0, f32_mma=1), 2),    # 3xTF32 up to D = 64 only
    (dict(D=128, in_dtype=0, f32_mma=1), 2),
    # K and V of 2^59 bytes each: refused before any size is computed in size_t
    (dict(B=1024, H=1024, HKV=1024, Sq=1, Sk=1 << 30), 1),
])
def test_invalid_params_rejected(fa, kw, code):
    p = _params(fa, **kw)
    assert fa.fa_fwd(A, A, A, A, A, p, 0) == code
    assert fa.fa_bwd(A, A, A, A, A, A, A, A, A, p, 0) == code
    assert fa.fa_bwd_dsmat(A, A, A, A, A, A, A, A, A, p, 0) == code


def test_materialised_ds_backward_is_bf16_only(fa):
    p = _params(fa, D=64, in_dtype=fa.FA_F32)
    assert fa.fa_bwd_dsmat(A, A, A, A, A, A, A, A, A, p, 0) == 2


def test_noalloc_rejects_oversized_params_before_sizing_scratch(fa):
    # a product of the shape fields that would wrap a size_t must not slip past the
    # scratch-size check
    p = _params(fa, B=1024, H=1024, HKV=1024, Sq=1, Sk=1 << 30)
    assert fa.fa_fwd_noalloc(A, A, A, A, A, p, 0) == 1


def test_null_params_rejected(fa):
    lib = fa.lib()
    assert lib.fa_fwd(A, A, A, A, A, None, None) == 1
    assert lib.fa_bwd(A, A, A, A, A, A, A, A, A, None, None) == 1


@pytest.mark.parametrize("which", range(5))
def test_fwd_null_and_misaligned_pointers(fa, which):
    p = _params(fa)
    ptrs = [A] * 5
    ptrs[which] = 0
    assert fa.fa_fwd(*ptrs, p, 0) == 1
    ptrs[which] = MIS
    assert fa.fa_fwd(*ptrs, p, 0) == 3


@pytest.mark.parametrize("which", range(9))
def test_bwd_null_and_misaligned_pointers(fa, which):
    p = _params(fa)
    ptrs = [A] * 9
    ptrs[which] = 0
    assert fa.fa_bwd(*ptrs, p, 0) == 1
    ptrs[which] = MIS
    assert fa.fa_bwd(*ptrs, p, 0) == 3


def test_empty_problems_are_no_ops(fa):
    # Sq == 0: nothing to compute, no pointer is touched and no CUDA call is made.
    assert fa.fa_fwd(0, 0, 0, 0, 0, _params(fa, Sq=0), 0) == 0
    assert fa.fa_bwd(0, 0, 0, 0, 0, 0, 0, 0, 0, _params(fa, Sq=0, Sk=0), 0) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    from attention_fa_fwd_02_gb300 import fa as fa_mod
    with pytest.raises(ImportError):
        fa_mod._load(str(tmp_path / "missing.so"))


def test_params_struct_layout_matches_the_header(fa, tmp_path):
    # the ctypes mirror of fa_params must have the C struct's size and field offsets
    import shutil
    import subprocess
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("needs gcc")
    names = [n for n, _ in fa.fa_params._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stddef.h>\n#include <stdio.h>\n#include \"fa.h\"\nint main(void) {\n"
                   + f'  printf("%zu", sizeof(fa_params));\n'
                   + "".join(f'  printf(" %zu", offsetof(fa_params, {n}));\n' for n in names)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(fa.fa_params)] + [getattr(fa.fa_params, n).offset for n in names]
    assert got == want
