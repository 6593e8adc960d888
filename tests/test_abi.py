"""The C ABI library builds, loads and exports every symbol include/rf.h
declares; host-side argument checks return their codes without a GPU.

These run on a CPU-only machine: every call below is rejected by the host
validation before any CUDA call is made.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from conftest import load_builder
    path = load_builder().build()
    return ctypes.CDLL(path)


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(rf_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("rf_attn_decode_split", "rf_state_merge", "rf_attn_prefill", "rf_softmax_topk",
              "rf_absmax_quant_fp8_gemm", "rf_status_string", "rf_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.rf_status_string.restype = ctypes.c_char_p
    assert lib.rf_status_string(0) == b"RF_OK"
    assert lib.rf_status_string(2) == b"RF_ERR_UNSUPPORTED"
    assert lib.rf_status_string(99) == b"RF_ERR_UNKNOWN"
    assert lib.rf_version() >= 10000


P = ctypes.c_void_p
FAKE = P(0x10000)          # aligned, never dereferenced: calls are rejected first
ODD = P(0x10004)           # 4-byte aligned only
NULL = P(0)
F = ctypes.c_float


def test_decode_fused_validation(lib):
    f = lib.rf_attn_decode_fused
    args = lambda **o: [o.get("q", FAKE), FAKE, FAKE, o.get("R", 4), o.get("L", 100), o.get("D", 128),
                        o.get("S", 4), F(o.get("scale", 0.1)), o.get("dtype", 1), FAKE, FAKE, FAKE,
                        o.get("counters", FAKE), o.get("out", FAKE), o.get("out_dtype", 1), NULL, NULL]
    assert f(*args(counters=NULL)) == 1
    assert f(*args(out=NULL)) == 1
    assert f(*args(out_dtype=5)) == 1
    assert f(*args(S=0)) == 1
    assert f(*args(D=64)) == 2            # bf16 with D=64 unsupported
    assert f(*args(counters=ODD)) == 3
    assert f(*args(out=ODD)) == 3


def test_decode_noalloc_validation(lib):
    # every refusal below comes from the host checks, before the call looks
    # up its static array or launches anything
    f = lib.rf_attn_decode_noalloc
    args = lambda **o: [o.get("q", FAKE), o.get("k", FAKE), o.get("v", FAKE), o.get("R", 4),
                        o.get("L", 100), o.get("D", 128), o.get("S", 4), F(o.get("scale", 0.1)),
                        o.get("dtype", 1), o.get("out", FAKE), o.get("out_dtype", 1), NULL, NULL]
    for name in ("q", "k", "v", "out"):
        assert f(*args(**{name: NULL})) == 1, name
    assert f(*args(dtype=7)) == 1
    assert f(*args(out_dtype=5)) == 1
    assert f(*args(S=0)) == 1
    assert f(*args(R=0)) == 1
    assert f(*args(L=-1)) == 1
    assert f(*args(scale=float("nan"))) == 1
    assert f(*args(scale=float("inf"))) == 1
    assert f(*args(D=64)) == 2              # bf16 with D=64 unsupported
    assert f(*args(D=128, dtype=0)) == 2    # fp32 with D=128 unsupported
    assert f(*args(R=1024, S=64)) == 2      # 34 MB of states > 16 MiB
    assert f(*args(R=65537, S=1, D=64, dtype=0)) == 2   # the size limit caps R at 65536
    for name in ("q", "k", "v", "out"):
        assert f(*args(**{name: ODD})) == 3, name


def test_decode_split_validation(lib):
    f = lib.rf_attn_decode_split
    args = lambda **o: [o.get("q", FAKE), FAKE, FAKE, o.get("R", 4), o.get("L", 100), o.get("D", 128),
                        o.get("S", 4), F(o.get("scale", 0.1)), o.get("dtype", 1),
                        FAKE, FAKE, o.get("acc", FAKE), NULL]
    assert f(*args(q=NULL)) == 1
    assert f(*args(R=0)) == 1
    assert f(*args(L=-1)) == 1
    assert f(*args(S=0)) == 1
    assert f(*args(scale=float("inf"))) == 1
    assert f(*args(dtype=7)) == 1
    assert f(*args(D=64)) == 2            # bf16 with D=64 unsupported
    assert f(*args(dtype=0)) == 2         # fp32 with D=128 unsupported
    assert f(*args(q=ODD)) == 3
    assert f(*args(acc=ODD)) == 3


def test_merge_validation(lib):
    f = lib.rf_state_merge
    base = dict(m=FAKE, R=4, S=8, D=128, out=FAKE, od=1)
    args = lambda **o: [o.get("m", FAKE), FAKE, o.get("acc", FAKE), o.get("R", 4), o.get("S", 8),
                        o.get("D", 128), o.get("out", FAKE), o.get("od", 1), NULL, NULL]
    assert f(*args(m=NULL)) == 1
    assert f(*args(out=NULL)) == 1
    assert f(*args(S=0)) == 1
    assert f(*args(od=5)) == 1
    assert f(*args(D=96)) == 2
    assert f(*args(out=ODD)) == 3
    assert base


def test_topk_validation(lib):
    f = lib.rf_softmax_topk
    args = lambda **o: [o.get("x", FAKE), o.get("T", 10), o.get("E", 64), o.get("k", 2), 1,
                        o.get("idx", FAKE), o.get("w", FAKE), NULL]
    assert f(*args(x=NULL)) == 1
    assert f(*args(idx=NULL)) == 1
    assert f(*args(w=NULL)) == 1
    assert f(*args(T=0)) == 1
    assert f(*args(k=0)) == 1
    assert f(*args(k=65)) == 1            # k > E
    assert f(*args(E=2048, k=4)) == 2
    assert f(*args(E=100, k=40)) == 2     # k > 32
    assert f(*args(x=ODD)) == 3
    assert f(*args(idx=ODD)) == 3
    assert f(*args(w=ODD)) == 3


def test_stream_read_validation(lib):
    f = lib.rf_stream_read
    f.argtypes = [P, ctypes.c_size_t, P, P]
    assert f(NULL, 64, FAKE, NULL) == 1
    assert f(FAKE, 64, NULL, NULL) == 1
    assert f(FAKE, 0, FAKE, NULL) == 1
    assert f(FAKE, 40, FAKE, NULL) == 2     # not a multiple of 16 bytes
    assert f(ODD, 64, FAKE, NULL) == 3
    assert f(FAKE, 64, P(0x10002), NULL) == 3


def test_quant_gemm_validation(lib):
    f = lib.rf_absmax_quant_fp8_gemm
    args = lambda **o: [o.get("x", FAKE), o.get("M", 256), o.get("K", 512), FAKE,
                        o.get("sw", FAKE), o.get("N", 256), FAKE, FAKE, FAKE, NULL]
    # every call below is rejected before a launch (ragged M and N are
    # supported, so they are only combined with a rejected argument)
    assert f(*args(x=NULL)) == 1
    assert f(*args(M=0)) == 1
    assert f(*args(K=100)) == 2
    assert f(*args(K=40, N=100, M=100)) == 2
    assert f(*args(K=65552)) == 2
    assert f(*args(x=ODD)) == 3
    assert f(*args(sw=ODD, N=100)) == 3
    g = lib.rf_fp8_gemm_scaled
    assert g(FAKE, FAKE, FAKE, ODD, 100, 300, 64, FAKE, NULL) == 3
    assert g(FAKE, FAKE, FAKE, FAKE, 100, 300, 24, FAKE, NULL) == 2
    q = lib.rf_absmax_quant_e4m3
    assert q(NULL, 4, 64, FAKE, FAKE, NULL) == 1
    assert q(FAKE, 4, 60, FAKE, FAKE, NULL) == 2
    assert q(ODD, 4, 64, FAKE, FAKE, NULL) == 3


def test_prefill_validation(lib):
    f = lib.rf_attn_prefill
    args = lambda **o: [FAKE, FAKE, FAKE, o.get("B", 1), 2, o.get("N", 256), o.get("D", 128), 1,
                        F(0.1), o.get("out", FAKE), NULL, NULL]
    assert f(*args(out=NULL)) == 1
    assert f(*args(B=0)) == 1
    assert f(*args(D=64)) == 2
    assert f(*args(B=1 << 20, N=4096)) == 2     # B*H*N rows past a 32-bit index
    assert f(*args(out=ODD)) == 3


def test_device_error_null(lib):
    assert lib.rf_device_error(NULL, NULL) == 1


def test_binding_declares_every_symbol():
    """The Python binding wraps every entry point the header declares."""
    import cascaded_reductions_gb300 as rf
    assert set(rf._SIGNATURES) == set(declared_symbols())


def test_row_cascade_validation(lib):
    sm = lib.rf_row_softmax
    assert sm(NULL, 4, 1024, FAKE, 1, NULL, NULL) == 1
    assert sm(FAKE, 0, 1024, FAKE, 1, NULL, NULL) == 1
    assert sm(FAKE, 4, 1024, FAKE, 7, NULL, NULL) == 1       # unknown level
    assert sm(FAKE, 4, 1024, FAKE, 0, NULL, NULL) == 1       # unfused needs work
    assert sm(FAKE, 4, 1022, FAKE, 1, NULL, NULL) == 2       # n % 4
    assert sm(FAKE, 4, 8196, FAKE, 3, NULL, NULL) == 2       # fused rows live in registers
    assert sm(ODD, 4, 1024, FAKE, 2, NULL, NULL) == 3
    var = lib.rf_row_variance
    assert var(FAKE, 4, 64, NULL, FAKE, 1, NULL) == 1
    assert var(FAKE, 4, 66, FAKE, FAKE, 1, NULL) == 2
    assert var(FAKE, 4, 64, FAKE, FAKE, -1, NULL) == 1
    moi = lib.rf_moment_of_inertia
    assert moi(FAKE, FAKE, 4, 64, FAKE, NULL, 1, NULL) == 1
    assert moi(FAKE, FAKE, 4, 6, FAKE, FAKE, 1, NULL) == 2
    assert moi(FAKE, ODD, 4, 64, FAKE, FAKE, 1, NULL) == 3


def test_layer_norm_validation(lib):
    ln = lib.rf_layer_norm
    args = lambda **o: [o.get("x", FAKE), FAKE, FAKE, o.get("R", 4), o.get("n", 64), F(o.get("eps", 1e-5)),
                        FAKE, o.get("level", 1), o.get("work", NULL), NULL]
    assert ln(*args(x=NULL)) == 1
    assert ln(*args(eps=-1.0)) == 1
    assert ln(*args(level=0)) == 1                    # unfused needs work
    assert ln(*args(n=66)) == 2
    assert ln(*args(n=8196)) == 2
    assert ln(*args(x=ODD)) == 3


def test_incremental_fp8_validation(lib):
    f = lib.rf_incremental_quant_fp8_gemm
    args = lambda **o: [o.get("x", FAKE), o.get("M", 128), o.get("K", 256), FAKE, FAKE,
                        o.get("N", 512), FAKE, NULL, NULL]
    assert f(*args(x=NULL)) == 1
    assert f(*args(M=0)) == 1
    assert f(*args(N=256)) == 2
    assert f(*args(K=100)) == 2
    assert f(*args(x=ODD)) == 3


def test_mla_decode_validation(lib):
    f = lib.rf_mla_decode_split
    args = lambda **o: [o.get("q", FAKE), o.get("c", FAKE), o.get("B", 2), o.get("H", 16),
                        o.get("L", 300), o.get("Dk", 576), o.get("Dv", 512), o.get("S", 4),
                        F(o.get("scale", 0.07)), FAKE, FAKE, o.get("acc", FAKE), NULL]
    assert f(*args(q=NULL)) == 1
    assert f(*args(c=NULL)) == 1
    assert f(*args(B=0)) == 1
    assert f(*args(L=0)) == 1
    assert f(*args(S=0)) == 1
    assert f(*args(scale=float("nan"))) == 1
    assert f(*args(Dk=512)) == 2
    assert f(*args(Dv=128)) == 2
    assert f(*args(H=8)) == 2
    assert f(*args(H=24)) == 2
    assert f(*args(B=70000, L=32768)) == 2     # B*L rows beyond a 32-bit TMA coordinate
    assert f(*args(q=ODD)) == 3
    assert f(*args(acc=ODD)) == 3


def test_merge_accepts_the_mla_value_width(lib):
    f = lib.rf_state_merge
    # D = 512 passes validation and fails only on the misaligned output
    assert f(FAKE, FAKE, FAKE, 4, 8, 512, ODD, 1, NULL, NULL) == 3


def test_selftest_validation(lib):
    assert lib.rf_selftest_wait_timeout(NULL, NULL) == 1


def test_rms_norm_validation(lib):
    f = lib.rf_rms_norm
    args = lambda **o: [o.get("x", FAKE), FAKE, o.get("R", 4), o.get("n", 64), F(o.get("eps", 1e-6)),
                        FAKE, o.get("level", 1), o.get("work", NULL), NULL]
    assert f(*args(x=NULL)) == 1
    assert f(*args(R=0)) == 1
    assert f(*args(eps=float("inf"))) == 1
    assert f(*args(level=7)) == 1
    assert f(*args(level=0)) == 1                    # unfused needs work
    assert f(*args(n=66)) == 2
    assert f(*args(n=8196)) == 2
    assert f(*args(x=ODD)) == 3
