"""Host-only tests of the C-ABI boundary: the library loads, exports every entry
point its header declares, and rejects bad arguments with the documented codes
before touching the GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import gated_deltanet_chunked_gdr_gb300 as gdr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(gdr_[A-Za-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_builds_and_exports_every_declared_symbol():
    lib = gdr.load_library()
    declared = _declared_functions()
    assert {"gdr_kkt_solve", "gdr_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert declared <= set(gdr.EXPORTED_SYMBOLS)


def _header_status_codes():
    text = open(os.path.join(ROOT, "include", "gdr_kkt_solve.h")).read()
    body = re.search(r"typedef enum \{(.*?)\} gdr_status;", text, flags=re.S).group(1)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(GDR_[A-Z0-9_]+)\s*=\s*(-?\d+)", body)}


def test_status_strings():
    codes = _header_status_codes()
    assert len(codes) == 11
    for name, code in codes.items():
        assert getattr(gdr, name) == code, name                 # binding constants = header enum
        s = gdr.status_string(code)
        assert isinstance(s, str) and s and s != "unknown gdr_status", name
    assert gdr.status_string(min(codes.values()) - 1) == "unknown gdr_status"
    assert gdr.status_string(-99) == "unknown gdr_status"


def test_status_strings_match_what_the_calls_accept():
    # The texts state the accepted set as the header does: chunk 128 for the
    # fused call, fp32 keys with K in {64, 128}, K <= 128 for those and chunk 128.
    chunk = gdr.status_string(gdr.GDR_ERR_CHUNK)
    assert "64" in chunk and "128" in chunk and "fused" in chunk
    dtype = gdr.status_string(gdr.GDR_ERR_DTYPE)
    assert "fp32" in dtype.split("beta")[0] and "{64, 128}" in dtype
    for t in ("bf16", "fp16"):
        assert t in dtype.split("beta")[0]
    shape = gdr.status_string(gdr.GDR_ERR_SHAPE)
    assert "{64, 128, 192, 256}" in shape and "K <= 128" in shape
    assert "cu[0] = 0" in gdr.status_string(gdr.GDR_ERR_CU_SEQLENS)
    assert "262144" in gdr.status_string(gdr.GDR_ERR_SCRATCH)


# Fake, well-aligned addresses: validation must fail before anything uses them.
K_PTR, OUT_PTR, G_PTR, B_PTR, CU_PTR = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000


def _call(**kw):
    a = dict(k=K_PTR, g=G_PTR, beta=B_PTR, cu=0, B=2, T=100, H=3, K=128, chunk=64,
             dtype=gdr.GDR_F32, out=OUT_PTR)
    a.update(kw)
    return gdr.kkt_solve_raw(a["k"], a["g"], a["beta"], a["cu"], a["B"], a["T"], a["H"], a["K"],
                             a["chunk"], a["dtype"], a["out"], 0)


@pytest.mark.parametrize("chunk", [0, 16, 32, 63, 65, 96, 256])
def test_chunk_size_must_be_64_or_128(chunk):
    assert _call(chunk=chunk) == gdr.GDR_ERR_CHUNK


def test_chunk_128_limits():
    import torch
    assert _call(chunk=128, K=192) == gdr.GDR_ERR_SHAPE          # chunk 128 takes K <= 128
    assert _call_kkt(chunk=128) == gdr.GDR_ERR_CHUNK             # the unfused chain is chunk 64 only
    assert _call_solve(chunk=128) == gdr.GDR_ERR_CHUNK
    assert _call_noalloc(chunk=128) == gdr.GDR_ERR_CHUNK
    if not torch.cuda.is_available():
        assert _call(chunk=128) == gdr.GDR_ERR_DEVICE
        assert _call(chunk=128, K=64) == gdr.GDR_ERR_DEVICE


@pytest.mark.parametrize("dtype", [-1, 3, 7])
def test_bad_out_dtype(dtype):
    assert _call(dtype=dtype) == gdr.GDR_ERR_DTYPE


def _call_ex(**kw):
    a = dict(k=K_PTR, kd=gdr.GDR_BF16, g=G_PTR, beta=B_PTR, bd=gdr.GDR_BF16, cu=0, B=2, T=100, H=3,
             K=128, chunk=64, dtype=gdr.GDR_F32, out=OUT_PTR)
    a.update(kw)
    return gdr.kkt_solve_ex_raw(a["k"], a["kd"], a["g"], a["beta"], a["bd"], a["cu"], a["B"], a["T"],
                                a["H"], a["K"], a["chunk"], a["dtype"], a["out"], 0)


@pytest.mark.parametrize("kw", [dict(kd=3), dict(kd=-1), dict(bd=3), dict(bd=-1), dict(dtype=3)])
def test_ex_bad_dtypes(kw):
    assert _call_ex(**kw) == gdr.GDR_ERR_DTYPE


def test_ex_fp32_key_limits():
    import torch
    assert _call_ex(kd=gdr.GDR_F32, K=192) == gdr.GDR_ERR_SHAPE       # fp32 keys: K <= 128
    assert _call_ex(kd=gdr.GDR_F32, chunk=128) == gdr.GDR_ERR_DTYPE  # and chunk 64 only
    assert _call_kkt(kd=gdr.GDR_F32) == gdr.GDR_ERR_DTYPE            # the chain takes 16-bit keys
    if not torch.cuda.is_available():
        assert _call_ex(kd=gdr.GDR_F32) == gdr.GDR_ERR_DEVICE
        assert _call_ex(kd=gdr.GDR_F32, K=64) == gdr.GDR_ERR_DEVICE


def test_ex_beta_dtype_ignored_without_beta():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call_ex(beta=0, bd=99) == gdr.GDR_ERR_DEVICE


@pytest.mark.parametrize("kw", [dict(beta=B_PTR + 2, bd=gdr.GDR_F32), dict(beta=B_PTR + 1, bd=gdr.GDR_F16),
                                dict(k=K_PTR + 8, kd=gdr.GDR_F16)])
def test_ex_misaligned(kw):
    assert _call_ex(**kw) == gdr.GDR_ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(K=64), dict(K=192), dict(K=256), dict(kd=gdr.GDR_F16),
                                dict(bd=gdr.GDR_F32), dict(bd=gdr.GDR_F16), dict(dtype=gdr.GDR_F16),
                                dict(beta=B_PTR + 2, bd=gdr.GDR_F16)])
def test_ex_valid_arguments_reach_the_device_check(kw):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call_ex(**kw) == gdr.GDR_ERR_DEVICE


@pytest.mark.parametrize("kw", [dict(K=0), dict(K=32), dict(K=127), dict(K=320), dict(B=-1), dict(T=-5),
                                dict(H=-2), dict(B=1 << 20, T=1 << 12),
                                dict(cu=CU_PTR, B=4, T=1 << 31)])
def test_bad_shapes(kw):
    assert _call(**kw) == gdr.GDR_ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(B=0), dict(T=0), dict(H=0), dict(B=0, k=0, out=0)])
def test_empty_problem_is_ok_and_launches_nothing(kw):
    assert _call(**kw) == gdr.GDR_OK


@pytest.mark.parametrize("kw", [dict(k=0), dict(out=0)])
def test_null_pointers(kw):
    assert _call(**kw) == gdr.GDR_ERR_NULL


@pytest.mark.parametrize("kw", [dict(k=K_PTR + 8), dict(out=OUT_PTR + 4), dict(g=G_PTR + 2),
                                dict(beta=B_PTR + 1), dict(cu=CU_PTR + 2)])
def test_misaligned_pointers(kw):
    assert _call(**kw) == gdr.GDR_ERR_ALIGN


def test_valid_arguments_without_gpu_report_device_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call() == gdr.GDR_ERR_DEVICE
    assert gdr.load_library().gdr_kkt_solve_num_sms() == gdr.GDR_ERR_DEVICE


def test_python_binding_rejects_chunk_size_like_the_page_api():
    import torch
    k = torch.zeros(1, 64, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdr.kkt_solve(k, chunk_size=32)
    with pytest.raises(ValueError):
        gdr.solve_tril(torch.zeros(1, 64, 1, 64), chunk_size=128)
    with pytest.raises(TypeError):
        gdr.kkt_solve(k)                       # CPU tensor: no CPU fallback exists


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "gated_deltanet_chunked_gdr_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "oracle_kkt_solve" not in text, fn


def _call_kkt(**kw):
    a = dict(k=K_PTR, kd=gdr.GDR_BF16, g=G_PTR, beta=B_PTR, bd=gdr.GDR_BF16, cu=0, B=2, T=100, H=3,
             K=128, chunk=64, A=OUT_PTR)
    a.update(kw)
    return gdr.chunk_scaled_dot_kkt_raw(a["k"], a["kd"], a["g"], a["beta"], a["bd"], a["cu"], a["B"],
                                        a["T"], a["H"], a["K"], a["chunk"], a["A"], 0)


def _call_solve(**kw):
    a = dict(A=K_PTR, cu=0, B=2, T=100, H=3, chunk=64, dtype=gdr.GDR_F32, out=OUT_PTR)
    a.update(kw)
    return gdr.solve_tril_raw(a["A"], a["cu"], a["B"], a["T"], a["H"], a["chunk"], a["dtype"],
                              a["out"], 0)


@pytest.mark.parametrize("call,kw,want", [
    (_call_kkt, dict(chunk=32), gdr.GDR_ERR_CHUNK), (_call_kkt, dict(A=0), gdr.GDR_ERR_NULL),
    (_call_kkt, dict(A=OUT_PTR + 4), gdr.GDR_ERR_ALIGN), (_call_kkt, dict(kd=gdr.GDR_F32), gdr.GDR_ERR_DTYPE),
    (_call_kkt, dict(K=96), gdr.GDR_ERR_SHAPE), (_call_kkt, dict(B=0), gdr.GDR_OK),
    (_call_solve, dict(chunk=128), gdr.GDR_ERR_CHUNK), (_call_solve, dict(A=0), gdr.GDR_ERR_NULL),
    (_call_solve, dict(out=0), gdr.GDR_ERR_NULL), (_call_solve, dict(A=K_PTR + 8), gdr.GDR_ERR_ALIGN),
    (_call_solve, dict(dtype=5), gdr.GDR_ERR_DTYPE), (_call_solve, dict(T=-1), gdr.GDR_ERR_SHAPE),
    (_call_solve, dict(H=0), gdr.GDR_OK)])
def test_unfused_chain_argument_checks(call, kw, want):
    assert call(**kw) == want


def test_unfused_chain_valid_arguments_reach_the_device_check():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call_kkt() == gdr.GDR_ERR_DEVICE
    assert _call_solve() == gdr.GDR_ERR_DEVICE


def _call_noalloc(**kw):
    a = dict(k=K_PTR, kd=gdr.GDR_BF16, g=G_PTR, beta=B_PTR, bd=gdr.GDR_BF16, cu=0, B=2, T=100, H=3,
             K=128, chunk=64, dtype=gdr.GDR_F32, out=OUT_PTR)
    a.update(kw)
    return gdr.kkt_solve_unfused_noalloc_raw(a["k"], a["kd"], a["g"], a["beta"], a["bd"], a["cu"], a["B"],
                                             a["T"], a["H"], a["K"], a["chunk"], a["dtype"], a["out"], 0)


@pytest.mark.parametrize("kw,want", [
    (dict(B=1, T=1 << 16, H=5), gdr.GDR_ERR_SCRATCH),          # 327680 token-heads > 262144
    (dict(B=5, T=1 << 16, H=1), gdr.GDR_ERR_SCRATCH),
    (dict(cu=CU_PTR, B=3, T=70000, H=4), gdr.GDR_ERR_SCRATCH),
    (dict(chunk=32), gdr.GDR_ERR_CHUNK), (dict(out=0), gdr.GDR_ERR_NULL),
    (dict(out=OUT_PTR + 8), gdr.GDR_ERR_ALIGN), (dict(dtype=9), gdr.GDR_ERR_DTYPE),
    (dict(K=100), gdr.GDR_ERR_SHAPE), (dict(T=0), gdr.GDR_OK), (dict(H=-1), gdr.GDR_ERR_SHAPE),
    (dict(kd=gdr.GDR_F32), gdr.GDR_ERR_DTYPE), (dict(kd=gdr.GDR_F32, K=64), gdr.GDR_ERR_DTYPE),
    (dict(chunk=128), gdr.GDR_ERR_CHUNK)])
def test_noalloc_argument_checks_and_size_limit(kw, want):
    assert _call_noalloc(**kw) == want


def test_noalloc_within_limit_reaches_the_device_check():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call_noalloc(B=1, T=1 << 16, H=4) == gdr.GDR_ERR_DEVICE     # exactly 262144


# gdr_kkt_solve_host: host pointers (any readable host address works for the
# checks, which happen before anything is enqueued) and a device workspace.
HOST_BUF = ctypes.create_string_buffer(4096 + 256)
HOST_PTR = (ctypes.addressof(HOST_BUF) + 255) // 256 * 256
WS_PTR = 1 << 40                      # 256-byte aligned stand-in device address


def _call_host(**kw):
    a = dict(k=HOST_PTR, kd=gdr.GDR_BF16, g=HOST_PTR, beta=HOST_PTR, bd=gdr.GDR_BF16, cu=0, B=2, T=100, H=3,
             K=128, chunk=64, dtype=gdr.GDR_F32, out=HOST_PTR, ws=WS_PTR, wsb=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = gdr.kkt_solve_host_workspace_bytes(gdr.GDR_BF16, 2, 100, 3, 128, 64, gdr.GDR_F32)
    return gdr.kkt_solve_host_raw(a["k"], a["kd"], a["g"], a["beta"], a["bd"], a["cu"], a["B"], a["T"], a["H"],
                                  a["K"], a["chunk"], a["dtype"], a["out"], a["ws"], a["wsb"], 0)


def test_host_workspace_bytes():
    n = gdr.kkt_solve_host_workspace_bytes(gdr.GDR_BF16, 2, 16384, 32, 128, 64, gdr.GDR_BF16)
    tok_heads = 2 * 16384 * 32
    # k, g, beta (fp32 room), cu, out, each 256-byte aligned
    assert n >= tok_heads * (256 + 4 + 4 + 128) and n % 256 == 0
    assert n < tok_heads * (256 + 4 + 4 + 128) + 5 * 256 + 4 * 3
    with pytest.raises(gdr.GdrError):
        gdr.kkt_solve_host_workspace_bytes(gdr.GDR_BF16, 2, 16, 2, 100, 64, gdr.GDR_F32)
    with pytest.raises(gdr.GdrError):
        gdr.kkt_solve_host_workspace_bytes(7, 2, 16, 2, 128, 64, gdr.GDR_F32)


@pytest.mark.parametrize("kw,want", [
    (dict(k=0), gdr.GDR_ERR_NULL), (dict(out=0), gdr.GDR_ERR_NULL), (dict(ws=0), gdr.GDR_ERR_NULL),
    (dict(wsb=1024), gdr.GDR_ERR_SHAPE), (dict(ws=WS_PTR + 16), gdr.GDR_ERR_ALIGN),
    (dict(chunk=32), gdr.GDR_ERR_CHUNK), (dict(dtype=9), gdr.GDR_ERR_DTYPE), (dict(kd=9), gdr.GDR_ERR_DTYPE),
    (dict(K=100), gdr.GDR_ERR_SHAPE), (dict(H=-1), gdr.GDR_ERR_SHAPE),
    (dict(kd=gdr.GDR_F32, K=256), gdr.GDR_ERR_SHAPE), (dict(T=0), gdr.GDR_OK), (dict(B=0), gdr.GDR_OK)])
def test_host_entry_argument_checks(kw, want):
    assert _call_host(**kw) == want


def test_host_entry_valid_arguments_reach_the_device_check():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert _call_host() == gdr.GDR_ERR_DEVICE


def test_host_binding_rejects_device_tensors_and_bad_types():
    import torch
    k = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        gdr.kkt_solve_host(k, g=torch.zeros(1, 64, 2, dtype=torch.float16))          # g must be fp32
    with pytest.raises(TypeError):
        gdr.kkt_solve_host(k, cu_seqlens=torch.tensor([0, 64], dtype=torch.int64))  # cu_seqlens int32
    with pytest.raises(TypeError):
        gdr.kkt_solve_host(k.float().double())                                       # fp64 keys
    with pytest.raises(ValueError):
        gdr.kkt_solve_host(k, out=torch.empty(1, 64, 2, 32))                          # wrong out shape


@pytest.mark.parametrize("cu,B,T,want", [
    (0, 3, 100, gdr.GDR_ERR_NULL), (CU_PTR + 2, 3, 100, gdr.GDR_ERR_ALIGN),
    (CU_PTR, -1, 100, gdr.GDR_ERR_SHAPE), (CU_PTR, 3, -1, gdr.GDR_ERR_SHAPE),
    (CU_PTR, 1 << 31, 100, gdr.GDR_ERR_SHAPE)])
def test_check_cu_seqlens_argument_checks(cu, B, T, want):
    assert gdr.check_cu_seqlens_raw(cu, B, T, 0) == want


def test_check_cu_seqlens_valid_arguments_reach_the_device_check():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this test covers the no-device path")
    assert gdr.check_cu_seqlens_raw(CU_PTR, 3, 100, 0) == gdr.GDR_ERR_DEVICE
    assert gdr.check_cu_seqlens_raw(CU_PTR, 0, 0, 0) == gdr.GDR_ERR_DEVICE
    with pytest.raises(TypeError):
        gdr.check_cu_seqlens(torch.tensor([0, 5], dtype=torch.int32), 5)      # CPU tensor
