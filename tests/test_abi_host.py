"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/fp8blk.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8blk.h")


@pytest.fixture(scope="module")
def fp8blk():
    from block_scaled_fp8_bf16_gb300 import build
    build.build()
    import block_scaled_fp8_bf16_gb300 as m
    m._L()
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FP8BLK_API\s+[\w\s\*]+?\b(fp8blk_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ("fp8blk_quant_act", "fp8blk_gemm_w8a8", "fp8blk_gemm_w8a16", "fp8blk_gemv_w8a16"):
        assert n in names


def test_library_exports_every_declared_symbol(fp8blk):
    lib = ctypes.CDLL(fp8blk.LIB_PATH)
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(declared_symbols()) == set(fp8blk.EXPORTS)


def declared_arg_counts():
    text = open(HEADER).read()
    out = {}
    for m in re.finditer(r"FP8BLK_API\s+[\w\s\*]+?\b(fp8blk_\w+)\s*\(([^)]*)\)", text):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = len(params)
    return out


def test_binding_arg_counts_match_header(fp8blk):
    counts = declared_arg_counts()
    assert set(counts) == set(fp8blk.EXPORTS)
    for name, n in counts.items():
        assert len(fp8blk.EXPORTS[name][1]) == n, name


def test_no_other_dynamic_exports(fp8blk):
    out = subprocess.run(["nm", "-D", "--defined-only", fp8blk.LIB_PATH], capture_output=True, text=True).stdout
    ours = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("fp8blk")}
    assert ours == set(declared_symbols())


def test_no_cuda_driver_link_dependency(fp8blk):
    out = subprocess.run(["ldd", fp8blk.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libtorch" not in out


def test_constraints(fp8blk):
    c = fp8blk.fp8blk_query_constraints()
    assert c["abi_version"] == 3
    assert c["scale_block_k"] == 128 and c["scale_block_n"] == 128 and c["ue8m0_block"] == 32
    assert c["gemv_max_m"] == 16 and c["ptr_align_bytes"] == 16 and c["lds_multiple"] == 4


def test_status_strings(fp8blk):
    for s in range(9):
        assert len(fp8blk._L().fp8blk_status_string(s)) > 0
    assert fp8blk._L().fp8blk_status_string(99) == b"unknown status"


P = 1 << 20          # a 16-byte aligned fake pointer; never dereferenced
MIS = P + 4          # misaligned fake pointer


def call_w8a8(lib, a=P, lda=512, s=P, lds=16, b=P, ldb=512, bs=P, c=P, ldc=256, M=16, N=256, K=512, flags=0):
    return lib.fp8blk_gemm_w8a8(a, lda, s, lds, b, ldb, bs, c, ldc, M, N, K, flags, None)


def test_w8a8_argument_errors(fp8blk):
    lib = fp8blk._L()
    assert call_w8a8(lib, M=-1) == 1
    assert call_w8a8(lib, N=200) == 2
    assert call_w8a8(lib, K=500) == 2
    assert call_w8a8(lib, M=0) == 0                 # no-op, no device needed
    assert call_w8a8(lib, N=0) == 0
    assert call_w8a8(lib, c=None) == 1
    assert call_w8a8(lib, a=None) == 1
    assert call_w8a8(lib, lda=256) == 1             # lda < K
    assert call_w8a8(lib, lds=8) == 1               # lds < M
    assert call_w8a8(lib, ldc=128) == 1             # ldc < N
    assert call_w8a8(lib, a=MIS) == 3
    assert call_w8a8(lib, bs=MIS) == 3
    assert call_w8a8(lib, lda=520) == 3             # row pitch not 16 B
    assert call_w8a8(lib, lds=18) == 3
    assert call_w8a8(lib, ldc=260) == 3
    assert call_w8a8(lib, M=1 << 31) == 2
    assert call_w8a8(lib, flags=4) == 1             # unknown launch flag
    assert call_w8a8(lib, M=0, flags=1) == 0        # FP8BLK_FLAG_PDL is known
    assert call_w8a8(lib, M=0, flags=2) == 0        # FP8BLK_FLAG_OUT_F32 is known
    assert call_w8a8(lib, ldc=258, flags=2) == 3    # float32 rows need ldc * 4 % 16 == 0
    assert call_w8a8(lib, ldc=260) == 3             # bf16 rows need ldc * 2 % 16 == 0 ...
    assert call_w8a8(lib, ldc=260, flags=2) != 3    # ... which float32 rows of the same pitch meet


def test_w8a16_and_gemv_argument_errors(fp8blk):
    lib = fp8blk._L()

    def g(fn, x=P, ldx=512, b=P, ldb=512, sc=P, fmt=0, c=P, ldc=256, M=4, N=256, K=512, flags=0):
        return getattr(lib, fn)(x, ldx, b, ldb, sc, fmt, c, ldc, M, N, K, flags, None)

    for fn in ("fp8blk_gemm_w8a16", "fp8blk_gemv_w8a16"):
        assert g(fn, fmt=2) == 1
        assert g(fn, N=96) == 2
        assert g(fn, K=96) == 2
        assert g(fn, M=0) == 0
        assert g(fn, sc=None) == 1
        assert g(fn, ldx=256) == 1
        assert g(fn, x=MIS) == 3
        assert g(fn, ldx=516) == 3
        assert g(fn, ldb=520) == 3
        assert g(fn, flags=4) == 1
        assert g(fn, M=0, flags=1) == 0
    assert g("fp8blk_gemv_w8a16", M=17) == 2


def test_quant_argument_errors(fp8blk):
    lib = fp8blk._L()
    q = lambda x=P, M=16, K=512, ldx=512, a=P, lda=512, s=P, lds=16: lib.fp8blk_quant_act(x, M, K, ldx, a, lda, s, lds, None)
    assert q(M=-1) == 1
    assert q(K=100) == 2
    assert q(M=0) == 0
    assert q(s=None) == 1
    assert q(lds=15) == 1
    assert q(lds=18) == 3
    assert q(a=MIS) == 3
    w = lambda N=256, K=512, ldw=512, ldb=512: lib.fp8blk_quant_weight(P, N, K, ldw, P, ldb, P, None)
    assert w(N=100) == 2
    assert w(ldw=100) == 1
    v = lambda fmt=0, N=256, K=512, counts=P: lib.fp8blk_validate_weights(P, 512, P, fmt, N, K, counts, None)
    assert v(fmt=3) == 1
    assert v(counts=None) == 1
    assert v(N=64) == 2
    d = lambda n=256, e=0: lib.fp8blk_debug_decode_e4m3(P, n, e, P, None)
    assert d(n=6) == 1
    assert d(e=8) == 1
    assert d(e=-15) == 1
    g = lambda n=64, a=P, s=P, ds=P, y=P: lib.fp8blk_debug_group_scale(a, n, s, ds, y, None)
    assert g(n=-1) == 1
    assert g(n=0) == 0
    assert g(y=None) == 1
    assert g(a=None) == 1
    assert g(s=P + 2) == 3


def test_valid_call_without_gpu_reports_cuda_or_arch(fp8blk):
    """A well-formed call on a machine without an sm_103 device must fail
    with a CUDA/arch status, never succeed silently."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_w8a8(fp8blk._L()) in (4, 5)


def test_wait_timeout_diag_argument_errors(fp8blk):
    L = fp8blk._L()
    for bad in (0, 999, 100_000_001, -5):
        assert L.fp8blk_debug_wait_timeout(bad, None) == 1   # FP8BLK_ERR_INVALID_ARG, no device work


def test_stream_read_diag_argument_errors(fp8blk):
    L = fp8blk._L()
    r = lambda p=P, n=4096, sink=P: L.fp8blk_debug_stream_read(p, n, sink, None)
    assert r(n=-16) == 1
    assert r(n=100) == 1        # not a multiple of 16 bytes
    assert r(n=0) == 0
    assert r(p=None) == 1
    assert r(sink=None) == 1
    assert r(p=MIS) == 3
    assert r(sink=P + 2) == 3


def test_grouped_argument_errors(fp8blk):
    L = fp8blk._L()
    P = ctypes.c_void_p(16 * 1024)   # a fake, 16-byte aligned device address: never dereferenced on these paths

    def g(M=256, N=256, K=512, G=2, rg=P, lda=512, lds=256, ldb=512, ldc=256, flags=0):
        return L.fp8blk_gemm_w8a8_grouped(P, lda, P, lds, P, ldb, P, rg, G, P, ldc, M, N, K, flags, None)

    assert g(G=0) == 1                 # at least one group
    assert g(M=200) == 2               # M % 128 for grouped rows
    assert g(N=200) == 2
    assert g(rg=None) == 1             # the row groups are required
    assert g(rg=ctypes.c_void_p(16 * 1024 + 2)) == 3   # int32 alignment
    assert g(flags=4) == 1
    assert g(M=0) == 0 and g(N=0) == 0  # no-ops, no device needed


def test_fused_linear_argument_errors(fp8blk):
    L = fp8blk._L()
    P = ctypes.c_void_p(16 * 1024)

    def f(M=16, N=256, K=512, ldx=512, ldb=512, ldc=256, flags=0, x=P):
        return L.fp8blk_linear_w8a8(x, ldx, P, ldb, P, P, ldc, M, N, K, flags, None)

    assert f(M=33) == 2                # more token rows than the fused form takes
    assert f(N=200) == 2 and f(K=500) == 2
    assert f(M=-1) == 1 and f(flags=4) == 1
    assert f(ldx=256) == 1             # ldx < K
    assert f(x=None) == 1
    assert f(ldx=516) == 3             # bf16 rows of x must be 16-byte multiples
    assert f(M=0) == 0                 # no-op, no device needed


def test_ue8m0_w8a8_argument_errors(fp8blk):
    L = fp8blk._L()
    P = ctypes.c_void_p(16 * 1024)

    def q(M=16, K=512, ldx=512, lda=512, x=P, e=P):
        return L.fp8blk_quant_act_ue8m0(x, M, K, ldx, P, lda, e, None)

    assert q(M=-1) == 1
    assert q(K=96) == 2                 # K % 128
    assert q(M=0) == 0                  # no-op
    assert q(e=None) == 1
    assert q(lda=256) == 1              # lda < K
    assert q(e=ctypes.c_void_p(16 * 1024 + 8)) == 3
    assert q(x=ctypes.c_void_p(16 * 1024 + 8)) == 3
    assert q(ldx=516) == 3

    def w(N=256, K=512, eb=P, sf=P):
        return L.fp8blk_ue8m0_weight_sf(eb, N, K, sf, None)

    assert w(N=96) == 2 and w(K=96) == 2
    assert w(N=-128) == 1
    assert w(N=0) == 0 and w(K=0) == 0  # no-ops
    assert w(eb=None) == 1 and w(sf=None) == 1
    assert w(sf=ctypes.c_void_p(16 * 1024 + 4)) == 3

    def g(M=16, N=256, K=512, lda=512, ldb=512, ldc=256, flags=0, ea=P, eb=P, c=P):
        return L.fp8blk_gemm_w8a8_ue8m0(P, lda, ea, P, ldb, eb, c, ldc, M, N, K, flags, None)

    assert g(N=96) == 2 and g(K=96) == 2
    assert g(M=-1) == 1 and g(flags=4) == 1
    assert g(M=0) == 0 and g(N=0) == 0  # no-ops, no device needed
    assert g(ea=None) == 1 and g(eb=None) == 1 and g(c=None) == 1
    assert g(ldb=256) == 1              # ldb < K
    assert g(eb=ctypes.c_void_p(16 * 1024 + 4)) == 3
    assert g(ldc=260) == 3              # bf16 rows need ldc * 2 % 16 == 0
    assert g(ldc=260, flags=2) != 3     # float32 rows of that pitch are fine


def test_ue8m0_sf_bytes(fp8blk):
    L = fp8blk._L()
    assert L.fp8blk_ue8m0_sf_bytes(1, 128) == 512
    assert L.fp8blk_ue8m0_sf_bytes(128, 128) == 512
    assert L.fp8blk_ue8m0_sf_bytes(129, 384) == 2 * 3 * 512
    assert L.fp8blk_ue8m0_sf_bytes(4096, 7168) == 32 * 56 * 512
    assert L.fp8blk_ue8m0_sf_bytes(0, 512) == 0
    assert L.fp8blk_ue8m0_sf_bytes(5, 0) == 0
    assert L.fp8blk_ue8m0_sf_bytes(-1, 128) == -1
    assert L.fp8blk_ue8m0_sf_bytes(16, 96) == -1
    assert L.fp8blk_ue8m0_sf_bytes(1 << 62, 1 << 20) == -1   # overflow


@pytest.mark.parametrize("rows,K", [(1, 128), (128, 256), (200, 384), (300, 1024)])
def test_ue8m0_tiled_layout_helpers(fp8blk, rows, K):
    """The binding's layout helpers against the byte offset stated for the
    tiled scale layout, written out element by element."""
    import torch
    rng = np.random.default_rng(rows + K)
    e = rng.integers(0, 255, size=(rows, K // 32), dtype=np.uint8)
    sf = fp8blk.ue8m0_sf_from_rows(torch.from_numpy(e), pad=0xEE).numpy()
    R, KB = (rows + 127) // 128, K // 128
    assert sf.size == R * KB * 512 == fp8blk.fp8blk_ue8m0_sf_bytes(rows, K)
    expect = np.full(sf.size, 0xEE, dtype=np.uint8)
    for r in range(rows):
        for g in range(K // 32):
            expect[((r // 128) * KB + g // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + g % 4] = e[r, g]
    assert np.array_equal(sf, expect)
    back = fp8blk.ue8m0_sf_to_rows(torch.from_numpy(sf), rows, K).numpy()
    assert np.array_equal(back, e)


def test_linear_fused_rule(fp8blk):
    """The binding's choice between the one-launch quantising W8A8 kernel and
    quant + GEMM (taken from measured rows of both forms)."""
    pdl = fp8blk.FLAG_PDL
    pref = fp8blk.linear_fused_preferred
    assert pref(16, 256, 512) and pref(32, 256, 512)            # small layers: one launch at every M <= 32
    assert pref(1, 4096, 4096) and pref(2, 2048, 7168)
    assert pref(4, 2048, 7168, pdl) and not pref(4, 2048, 7168)
    assert pref(8, 4096, 4096) and not pref(8, 4096, 4096, pdl)
    assert pref(8, 7168, 2048, pdl) and not pref(8, 2048, 7168)
    assert not pref(16, 4096, 4096) and not pref(32, 7168, 2048, pdl)
    assert not pref(33, 256, 512) and not pref(0, 256, 512)
