"""The C-ABI library loads and exports every symbol the header declares; host-side argument
checks that need no GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from routed_moe_fp4_gb300 import build, colimoe
    build.build()
    return colimoe.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "colimoe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"COLI_API[^;(]*?\b(coli_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    assert {"coli_moe_create", "coli_moe_forward", "coli_moe_destroy"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    from routed_moe_fp4_gb300 import colimoe
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(colimoe.EXPORTED)


def test_create_rejects_bad_config(lib):
    from routed_moe_fp4_gb300 import colimoe as cm
    bad = [
        cm.coli_moe_config(0, 256, 128, 128, 4, 2),       # E = 0
        cm.coli_moe_config(8, 200, 128, 128, 4, 2),       # H not a multiple of 128
        cm.coli_moe_config(8, 256, 96, 128, 4, 2),        # I not a multiple of 128
        cm.coli_moe_config(8, 256, 128, 100, 4, 2),       # I_s not a multiple of 128
        cm.coli_moe_config(8, 256, 128, 128, 0, 2),       # max_tokens = 0
        cm.coli_moe_config(8, 256, 128, 128, 4, 9),       # max_top_k > E
        cm.coli_moe_config(64, 256, 128, 128, 4, 33),     # max_top_k > 32
    ]
    for cfg in bad:
        out = C.c_void_p(1)
        rc = lib.coli_moe_create(C.byref(cfg), None, C.byref(out))
        assert rc == cm.COLI_ERR_INVALID_ARG
        assert out.value is None
        assert "invalid config" in cm.coli_moe_last_error(None)


def test_null_arguments(lib):
    from routed_moe_fp4_gb300 import colimoe as cm
    assert lib.coli_moe_create(None, None, None) == cm.COLI_ERR_INVALID_ARG
    lib.coli_moe_destroy(None)                       # no-op
    assert lib.coli_moe_set_ffn_path(None, 0) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_moe_forward(None, None, 0, None, None, None, None, 1, None) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_moe_last_launch_count(None) == 0
    assert isinstance(cm.coli_moe_last_error(None), str)


def test_create_without_gpu_is_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this host has a GPU")
    from routed_moe_fp4_gb300 import colimoe as cm
    cfg = cm.coli_moe_config(8, 256, 128, 128, 4, 2)
    out = C.c_void_p()
    rc = lib.coli_moe_create(C.byref(cfg), None, C.byref(out))
    assert rc == cm.COLI_ERR_UNSUPPORTED_ARCH and out.value is None


def test_null_arguments_of_the_bank_dense_and_nvfp4_calls(lib):
    from routed_moe_fp4_gb300 import colimoe as cm
    out = C.c_void_p(1)
    assert lib.coli_bank_create(None, 4, None, C.byref(out)) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_bank_create(None, 4, None, None) == cm.COLI_ERR_INVALID_ARG
    lib.coli_bank_destroy(None)                      # no-op
    assert lib.coli_bank_set_copy_blocks(None, 4) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_bank_state(None, None, None, None, None, None) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_moe_forward_banked(None, None, None, 1, None, None, None, 1, None) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_moe_forward_nvfp4(None, None, 1, None, None, None, None, 1, None) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_dense_create(4, 256, None, None) == cm.COLI_ERR_INVALID_ARG
    assert lib.coli_dense_forward(None, None, 1, 128, None, None, 128, None) == cm.COLI_ERR_INVALID_ARG
    lib.coli_dense_destroy(None)                     # no-op
    code = C.c_int32(0)
    assert lib.coli_dense_device_error(None, C.byref(code)) == cm.COLI_ERR_INVALID_ARG
    assert isinstance(cm.coli_dense_last_error(None), str)


def test_dense_create_rejects_bad_sizes(lib):
    from routed_moe_fp4_gb300 import colimoe as cm
    for max_tokens, max_k in ((0, 256), (4, 100), (4, 0), (4, 64)):
        out = C.c_void_p(1)
        assert lib.coli_dense_create(max_tokens, max_k, None, C.byref(out)) == cm.COLI_ERR_INVALID_ARG
        assert out.value is None
        assert "invalid dense config" in cm.coli_dense_last_error(None)


def test_dense_create_without_gpu_is_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this host has a GPU")
    from routed_moe_fp4_gb300 import colimoe as cm
    out = C.c_void_p()
    assert lib.coli_dense_create(4, 256, None, C.byref(out)) == cm.COLI_ERR_UNSUPPORTED_ARCH
    assert out.value is None


def test_binding_refuses_strided_views():
    import numpy as np
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    t = torch.zeros((8, 16), dtype=torch.int16)
    assert cm._ptr(t) == t.data_ptr() and cm._ptr(t[2:5]) == t[2:5].data_ptr()
    with pytest.raises(ValueError):
        cm._ptr(t.t())
    with pytest.raises(ValueError):
        cm._ptr(t[:, ::2])
    a = np.zeros((8, 16), np.uint8)
    assert cm._ptr(a) == a.ctypes.data
    with pytest.raises(ValueError):
        cm._ptr(a[:, 1:])
    assert cm._ptr(None) is None and cm._ptr(1234) == 1234


def test_header_is_plain_c_with_only_stdint(tmp_path):
    """The ABI header includes only <stdint.h> and compiles as strict C99 and as C++."""
    import shutil
    import subprocess
    hdr = os.path.join(ROOT, "include", "colimoe.h")
    with open(hdr) as f:
        includes = re.findall(r"^\s*#\s*include\s*[<\"]([^>\"]+)[>\"]", f.read(), re.M)
    assert includes == ["stdint.h"]
    src = tmp_path / "use.c"
    src.write_text('#include "colimoe.h"\nint main(void) { coli_moe_config c = {1, 128, 128, 0, 1, 1}; (void)c;'
                   ' const char *(*f)(const coli_moe_t *) = coli_moe_last_error; (void)f; return 0; }\n')
    for cc, std in (("gcc", "-std=c99"), ("g++", "-std=c++17")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not found")
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                            "-x", "c" if cc == "gcc" else "c++", f"-I{os.path.join(ROOT, 'include')}", str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_route_static_checks_arguments_before_the_device(lib):
    """Bad sizes, oversize scratch and NULL or misaligned pointers are rejected before any CUDA
    call; valid arguments without a GPU give an error code, never a host fallback."""
    from routed_moe_fp4_gb300 import colimoe as cm
    lib_fn = lib.coli_moe_route_static
    buf = (C.c_uint8 * 4096)()
    base = (C.addressof(buf) + 15) & ~15                 # a 16-byte aligned host address
    good = dict(x=base, T=4, H=256, w=base, b=None, E=8, k=2, idx=base, wt=base)

    def call(**kw):
        a = dict(good, **kw)
        return lib_fn(a["x"], a["T"], a["H"], a["w"], a["b"], a["E"], a["k"], a["idx"], a["wt"], None)

    assert call(T=0) == cm.COLI_OK                        # nothing to do
    for bad in (dict(T=-1), dict(E=0), dict(E=1025), dict(H=100), dict(H=0), dict(k=0), dict(k=9),
                dict(k=33, E=64), dict(T=2048, E=256), dict(x=None), dict(w=None), dict(idx=None),
                dict(wt=None), dict(x=base + 2), dict(w=base + 4)):
        assert call(**bad) == cm.COLI_ERR_INVALID_ARG, bad
        assert "route_static" in cm.coli_moe_last_error(None)
    assert "scratch limit" in (call(T=2048, E=256), cm.coli_moe_last_error(None))[1]
    import torch
    if not torch.cuda.is_available():
        assert call() in (cm.COLI_ERR_CUDA, cm.COLI_ERR_UNSUPPORTED_ARCH)


def test_create_frees_everything_when_any_allocation_fails():
    """The workspace allocation of coli_moe_create, run on a host allocator that fails at each
    allocation in turn: every failure returns COLI_ERR_OUT_OF_MEMORY with nothing left allocated,
    and the sequence without a failure completes and frees every block."""
    from routed_moe_fp4_gb300 import build, colimoe as cm
    build.build()
    for cfg in (cm.coli_moe_config(256, 4096, 2048, 2048, 8, 8), cm.coli_moe_config(8, 256, 128, 0, 1, 2)):
        rc, n, live = cm.coli_moe_test_alloc_failure(cfg, -1)
        assert rc == cm.COLI_OK and live == 0 and n > 20
        for k in range(n):
            rc_k, n_k, live_k = cm.coli_moe_test_alloc_failure(cfg, k)
            assert rc_k == cm.COLI_ERR_OUT_OF_MEMORY, k
            assert n_k == k + 1, (k, n_k)        # nothing is allocated after the failing call
            assert live_k == 0, (k, live_k)       # everything allocated before it was freed
        rc, n2, live = cm.coli_moe_test_alloc_failure(cfg, n)
        assert rc == cm.COLI_OK and n2 == n and live == 0
    bad = cm.coli_moe_config(0, 4096, 2048, 2048, 8, 8)
    assert cm.coli_moe_test_alloc_failure(bad, 0)[0] == cm.COLI_ERR_INVALID_ARG
