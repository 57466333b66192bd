"""The C ABI without a GPU: the library builds and loads, it exports every
entry point include/bil.h declares, and its host-side argument checks reject
bad calls before anything touches CUDA."""
import ctypes
import os
import re

import pytest

from invariant_token_log_gb300 import _lib
from invariant_token_log_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bil.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bil_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_operator_calls():
    names = declared_functions()
    for n in ("bil_logp_fwd", "bil_logp_bwd", "bil_logp_tile_partials", "bil_logp_merge"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict(re.findall(r"#define (BIL_[A-Z_0-9]+) \(?([0-9]+(?: \* 1024)?)\)?", text))
    assert int(consts["BIL_OK"]) == _lib.OK
    assert int(consts["BIL_E_TARGET_RANGE"]) == _lib.E_TARGET_RANGE
    assert int(consts["BIL_E_UNSUPPORTED"]) == _lib.E_UNSUPPORTED
    assert (int(consts["BIL_F32"]), int(consts["BIL_BF16"]), int(consts["BIL_F16"])) == (_lib.F32, _lib.BF16, _lib.F16)
    assert eval(consts["BIL_MAX_TILE_BYTES"]) == _lib.MAX_TILE_BYTES
    assert int(consts["BIL_MAX_FUSED_TILES"]) == _lib.MAX_FUSED_TILES
    assert re.search(r"#define BIL_MAX_EXTENT_BYTES \(\(int64_t\)1 << 48\)", text)
    assert _lib.MAX_EXTENT_BYTES == 2 ** 48


def test_contract_id_and_status_strings(lib):
    cid = _lib.contract_id()
    assert cid.startswith("bil.v4") and "ex2.approx" in cid and "fma" in cid and "entropy" in cid
    for s in range(7):
        assert _lib.status_string(s) != "unknown status"
    assert _lib.status_string(99) == "unknown status"


# Bad arguments are rejected on the host, before any CUDA call, so these run
# without a GPU.  A fake non-null device pointer is never dereferenced.
FAKE = ctypes.c_void_p(0x10000)
FAKE_ODD = ctypes.c_void_p(0x10001)
NULL = None


def fwd(lib, **kw):
    a = dict(logits=FAKE, dtype=_lib.BF16, n=4, vocab=300, ld=300, tgt=FAKE, ign=-100, tile=4096, temp=1.0,
             logp=FAKE, lse=FAKE, ent=NULL, validate=0, stream=NULL)
    a.update(kw)
    return lib.bil_logp_fwd(a["logits"], a["dtype"], a["n"], a["vocab"], a["ld"], a["tgt"], a["ign"], a["tile"],
                            a["temp"], a["logp"], a["lse"], a["ent"], a["validate"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), _lib.E_INVALID_ARG),
    (dict(vocab=0), _lib.E_INVALID_ARG),
    (dict(ld=299), _lib.E_INVALID_ARG),
    (dict(dtype=7), _lib.E_DTYPE),
    (dict(tile=0), _lib.E_INVALID_ARG),
    (dict(tile=12), _lib.E_INVALID_ARG),
    (dict(tile=65536), _lib.E_UNSUPPORTED),
    (dict(dtype=_lib.F32, tile=32768), _lib.E_UNSUPPORTED),
    (dict(temp=0.0), _lib.E_INVALID_ARG),
    (dict(temp=-1.0), _lib.E_INVALID_ARG),
    (dict(temp=float("nan")), _lib.E_INVALID_ARG),
    (dict(temp=float("inf")), _lib.E_INVALID_ARG),
    (dict(temp=1e-45), _lib.E_INVALID_ARG),
    (dict(logits=NULL), _lib.E_INVALID_ARG),
    (dict(tgt=NULL), _lib.E_INVALID_ARG),
    (dict(logp=NULL), _lib.E_INVALID_ARG),
    (dict(logits=FAKE_ODD), _lib.E_ALIGN),
    (dict(tgt=ctypes.c_void_p(0x10004)), _lib.E_ALIGN),
    (dict(ent=FAKE_ODD), _lib.E_ALIGN),
    (dict(vocab=8 * 2049, ld=8 * 2049, tile=8), _lib.E_UNSUPPORTED),
    # rows x pitch x element size above 2^48 bytes; exactly 2^48 passes the extent check
    (dict(n=2 ** 20, vocab=300, ld=2 ** 27 + 8), _lib.E_UNSUPPORTED),
    (dict(n=2 ** 40, vocab=300, ld=304), _lib.E_UNSUPPORTED),
    (dict(n=2 ** 62, vocab=300, ld=300), _lib.E_UNSUPPORTED),
    (dict(n=2 ** 20, vocab=300, ld=2 ** 27, logits=NULL), _lib.E_INVALID_ARG),
    (dict(vocab=2 ** 48 + 1, ld=2 ** 48 + 1), _lib.E_UNSUPPORTED),
    (dict(vocab=2 ** 63 - 1, ld=2 ** 63 - 1), _lib.E_UNSUPPORTED),
    (dict(n=0), _lib.OK),
    (dict(n=0, logits=NULL, tgt=NULL, logp=NULL), _lib.OK),
])
def test_fwd_rejects_bad_arguments(lib, kw, status):
    assert fwd(lib, **kw) == status


def test_partials_rejects_bad_ranges(lib):
    def call(**kw):
        a = dict(n=4, vocab=10000, ld=10000, tile=4096, b=0, e=3, ldp=3, temp=1.0, pe=NULL)
        a.update(kw)
        return lib.bil_logp_tile_partials(FAKE, _lib.BF16, a["n"], a["vocab"], a["ld"], a["tile"], a["b"], a["e"],
                                          a["temp"], FAKE, -100, FAKE, FAKE, a["pe"], a["ldp"], FAKE, NULL)
    assert call(b=-1) == _lib.E_INVALID_ARG
    assert call(b=2, e=2) == _lib.E_INVALID_ARG
    assert call(e=4) == _lib.E_INVALID_ARG          # only 3 tiles exist
    assert call(ldp=2) == _lib.E_INVALID_ARG
    assert call(b=1, e=3, ld=10000 - 4096 - 1) == _lib.E_INVALID_ARG  # shard narrower than its columns
    assert call(temp=0.0) == _lib.E_INVALID_ARG
    assert call(pe=FAKE_ODD) == _lib.E_ALIGN
    assert call(n=0) == _lib.OK
    assert call(n=2 ** 40) == _lib.E_UNSUPPORTED                       # logits extent above 2^48 bytes
    assert call(n=2 ** 20, ldp=2 ** 26 + 1) == _lib.E_UNSUPPORTED      # partials extent above 2^48 bytes
    assert call(vocab=2 ** 63 - 1, e=1, ld=4096) == _lib.E_UNSUPPORTED  # ceil(vocab / tile) cannot overflow


def test_merge_and_bwd_reject_bad_arguments(lib):
    m = lib.bil_logp_merge
    #   part_max part_sum part_ent n  T  ld tl    tgt   ign  V   logp  lse   ent   val stream
    assert m(FAKE, FAKE, NULL, 4, 0, 1, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == _lib.E_INVALID_ARG
    assert m(FAKE, FAKE, NULL, 4, 3, 2, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == _lib.E_INVALID_ARG
    assert m(FAKE, NULL, NULL, 4, 3, 3, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == _lib.E_INVALID_ARG
    assert m(FAKE_ODD, FAKE, NULL, 4, 3, 3, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == _lib.E_ALIGN
    # entropy output without entropy partials, and the other way round
    assert m(FAKE, FAKE, NULL, 4, 3, 3, FAKE, FAKE, -100, 10, FAKE, FAKE, FAKE, 0, NULL) == _lib.E_INVALID_ARG
    assert m(FAKE, FAKE, FAKE, 4, 3, 3, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == _lib.E_INVALID_ARG
    b = lib.bil_logp_bwd
    #       logits dtype      n  V    ld   tgt   ign  temp lse   g     ent   gent  d     odt        ldo  cols stream
    args = [FAKE, _lib.BF16, 4, 300, 300, FAKE, -100, 1.0, FAKE, FAKE, NULL, NULL, FAKE, _lib.BF16, 300, 300, NULL]

    def with_(**kw):
        a = list(args)
        for k, v in kw.items():
            a[{"odt": 13, "ldo": 14, "cols": 15, "d": 12, "temp": 7, "ent": 10, "gent": 11, "n": 2}[k]] = v
        return b(*a)
    assert with_(odt=9) == _lib.E_DTYPE
    assert with_(ldo=299, cols=299) == _lib.E_INVALID_ARG   # fewer output columns than vocab
    assert with_(ldo=300, cols=301) == _lib.E_INVALID_ARG   # out_cols beyond ld_out
    assert with_(d=FAKE_ODD) == _lib.E_ALIGN
    assert with_(temp=-2.0) == _lib.E_INVALID_ARG
    assert with_(ent=FAKE) == _lib.E_INVALID_ARG             # entropy without its gradient
    assert with_(gent=FAKE) == _lib.E_INVALID_ARG
    assert with_(n=0) == _lib.OK
    assert with_(n=2 ** 40) == _lib.E_UNSUPPORTED                          # input extent above 2^48 bytes
    assert with_(odt=_lib.F32, n=2 ** 20, ldo=2 ** 26 + 4) == _lib.E_UNSUPPORTED  # output extent
    assert m(FAKE, FAKE, NULL, 2 ** 40, 3, 2 ** 7, FAKE, FAKE, -100, 10, FAKE, FAKE, NULL, 0, NULL) == \
        _lib.E_UNSUPPORTED


def test_lm_head_calls_reject_extents_above_the_limit(lib):
    """The LM-head entries refuse buffers spanning more than 2^48 bytes, and
    vocabularies above it, on the host; these calls would otherwise reach a
    launch (a CUDA error without a GPU)."""
    big = _lib.MAX_EXTENT_BYTES
    out = ctypes.c_int64(0)
    ws = lib.bil_linear_logp_workspace_bytes
    assert ws(4, 1000, 0, ctypes.byref(out)) == _lib.OK
    part = -(-4 * 4 * 4 // 256) * 256       # [4 rows, 4 tiles of 256] float32, 256-byte aligned
    assert out.value == 2 * part + 256
    assert ws(2 ** 40, 151936, 0, ctypes.byref(out)) == _lib.E_UNSUPPORTED
    assert ws(4, 2 ** 63 - 1, 1, ctypes.byref(out)) == _lib.E_UNSUPPORTED
    assert ws(-1, 1000, 0, ctypes.byref(out)) == _lib.E_INVALID_ARG

    def partials(**kw):
        a = dict(n=4, ld_h=64, vocab=1000, ld_w=64, te=4, ldp=4, logits=NULL, ldl=0)
        a.update(kw)
        return lib.bil_linear_logp_partials(FAKE, FAKE, _lib.BF16, a["n"], 64, a["ld_h"], a["vocab"], a["ld_w"], 0,
                                            a["te"], 1.0, FAKE, -100, FAKE, FAKE, NULL, a["ldp"], FAKE, a["logits"],
                                            _lib.F32, a["ldl"], NULL)
    # the plain argument checks
    def partials_dt(dtype, **kw):
        a = dict(n=4, h=64, ld_h=64, vocab=1000, ld_w=64, tb=0, te=4, ldp=4, hidden=FAKE, logits=NULL,
                 ldt=_lib.F32, ldl=0)
        a.update(kw)
        return lib.bil_linear_logp_partials(a["hidden"], FAKE, dtype, a["n"], a["h"], a["ld_h"], a["vocab"],
                                            a["ld_w"], a["tb"], a["te"], 1.0, FAKE, -100, FAKE, FAKE, NULL, a["ldp"],
                                            FAKE, a["logits"], a["ldt"], a["ldl"], NULL)
    assert partials_dt(_lib.F32) == _lib.E_DTYPE                       # 16-bit operands only
    assert partials_dt(_lib.BF16, ld_h=63) == _lib.E_INVALID_ARG       # ld_hidden < hidden_size
    assert partials_dt(_lib.BF16, te=5) == _lib.E_INVALID_ARG          # 1000 columns are 4 tiles of 256
    assert partials_dt(_lib.BF16, tb=2, te=2) == _lib.E_INVALID_ARG
    assert partials_dt(_lib.BF16, ldp=3) == _lib.E_INVALID_ARG
    assert partials_dt(_lib.BF16, logits=FAKE, ldt=_lib.F16, ldl=1000) == _lib.E_DTYPE
    assert partials_dt(_lib.BF16, logits=FAKE, ldl=999) == _lib.E_INVALID_ARG
    assert partials_dt(_lib.BF16, hidden=ctypes.c_void_p(0x10008)) == _lib.E_ALIGN   # TMA: 16-byte base
    assert partials_dt(_lib.BF16, h=60, ld_h=60) == _lib.E_ALIGN        # TMA: 16-byte row stride
    assert partials_dt(_lib.F16, n=0) == _lib.OK
    assert partials(n=2 ** 20, ld_h=2 ** 30) == _lib.E_UNSUPPORTED                 # hidden: 2^51 bytes
    assert partials(ld_w=2 ** 40) == _lib.E_UNSUPPORTED                            # 1000 weight rows
    assert partials(n=2 ** 20, ldp=2 ** 27) == _lib.E_UNSUPPORTED                  # partials: 2^49 bytes
    assert partials(n=2 ** 20, logits=FAKE, ldl=2 ** 28) == _lib.E_UNSUPPORTED     # logits: 2^50 bytes
    assert partials(vocab=2 ** 63 - 1) == _lib.E_UNSUPPORTED
    assert partials(vocab=big + 1) == _lib.E_UNSUPPORTED

    def bwd_args(**kw):
        a = dict(dtype=_lib.BF16, n=4, vocab=1000, te=4, ent=NULL, gent=NULL, ld_dz=1000, dh_t=_lib.F32,
                 dw_t=_lib.F32, weight=FAKE, dweight=FAKE, dhidden=FAKE, dz=FAKE, ld_dh=64, ld_dw=64)
        a.update(kw)
        return lib.bil_linear_logp_bwd(FAKE, a["weight"], a["dtype"], a["n"], 64, 64, a["vocab"], 64, 0, a["te"],
                                       1.0, FAKE, -100, FAKE, FAKE, a["ent"], a["gent"], a["dz"], a["ld_dz"],
                                       a["dhidden"], a["dh_t"], a["ld_dh"], a["dweight"], a["dw_t"], a["ld_dw"], NULL)
    assert bwd_args(dtype=_lib.F32) == _lib.E_DTYPE
    assert bwd_args(dh_t=_lib.F16) == _lib.E_DTYPE             # outputs: float32 or the input type
    assert bwd_args(dw_t=_lib.F16) == _lib.E_DTYPE
    assert bwd_args(te=5) == _lib.E_INVALID_ARG                # beyond the 4 tiles of 1000 columns
    assert bwd_args(ld_dz=999) == _lib.E_INVALID_ARG           # dZ narrower than the shard
    assert bwd_args(ld_dh=63) == _lib.E_INVALID_ARG
    assert bwd_args(ld_dw=63) == _lib.E_INVALID_ARG
    assert bwd_args(ent=FAKE) == _lib.E_INVALID_ARG            # entropy without its gradient
    assert bwd_args(weight=NULL) == _lib.E_INVALID_ARG
    assert bwd_args(weight=ctypes.c_void_p(0x10008)) == _lib.E_ALIGN
    assert bwd_args(dz=NULL) == _lib.E_INVALID_ARG
    assert bwd_args(dhidden=NULL) == _lib.E_INVALID_ARG
    assert bwd_args(dweight=NULL) == _lib.E_INVALID_ARG
    assert bwd_args(dhidden=ctypes.c_void_p(0x10008)) == _lib.E_ALIGN
    assert bwd_args(dh_t=_lib.BF16, ld_dh=68) == _lib.E_ALIGN  # 136-byte rows of a 16-bit dhidden
    assert bwd_args(n=2 ** 20, ld_dz=2 ** 28) == _lib.E_UNSUPPORTED     # dZ: 2^49 bytes
    assert bwd_args(n=2 ** 20, ld_dh=2 ** 28) == _lib.E_UNSUPPORTED     # dhidden: 2^50 bytes
    assert bwd_args(ld_dw=2 ** 40) == _lib.E_UNSUPPORTED                # dweight
    assert bwd_args(vocab=2 ** 63 - 1) == _lib.E_UNSUPPORTED


def test_gemm_and_grad_check_their_arguments(lib):
    g = lib.bil_linear_gemm
    K, MN = _lib.LAYOUT_K_MAJOR, _lib.LAYOUT_MN_MAJOR
    ok = dict(a=FAKE, la=K, b=FAKE, lb=K, dt=_lib.BF16, m=4, n=8, k=64, lda=64, ldb=64, c=FAKE, ct=_lib.F32, ldc=8)

    def gemm(**kw):
        a = dict(ok)
        a.update(kw)
        return g(a["a"], a["la"], a["b"], a["lb"], a["dt"], a["m"], a["n"], a["k"], a["lda"], a["ldb"], a["c"],
                 a["ct"], a["ldc"], NULL)
    assert gemm(dt=_lib.F32) == _lib.E_DTYPE                     # 16-bit operands only
    assert gemm(ct=_lib.F16) == _lib.E_DTYPE                     # C: float32 or the operands' type
    assert gemm(la=2) == _lib.E_INVALID_ARG                      # a layout the header does not define
    assert gemm(lb=-1) == _lib.E_INVALID_ARG
    assert gemm(k=0) == _lib.E_INVALID_ARG
    assert gemm(lda=63) == _lib.E_INVALID_ARG                    # a K-major row holds k elements
    assert gemm(ldb=63) == _lib.E_INVALID_ARG
    assert gemm(la=MN, lda=3) == _lib.E_INVALID_ARG              # an MN-major row holds m ...
    assert gemm(lb=MN, ldb=7) == _lib.E_INVALID_ARG              # ... or n elements
    assert gemm(la=MN, lda=8, lb=MN, ldb=8, c=FAKE_ODD) == _lib.E_ALIGN  # [k, m], [k, n] rows pass; C's base fails
    assert gemm(ldc=7) == _lib.E_INVALID_ARG
    assert gemm(m=-1) == _lib.E_INVALID_ARG
    assert gemm(m=0, a=NULL, c=NULL) == _lib.OK                  # nothing to compute
    assert gemm(a=NULL) == _lib.E_INVALID_ARG
    assert gemm(a=ctypes.c_void_p(0x10008)) == _lib.E_ALIGN      # TMA: 16-byte base
    assert gemm(k=60, lda=60, ldb=64) == _lib.E_ALIGN            # TMA: 16-byte row stride
    assert gemm(la=MN, lda=4) == _lib.E_ALIGN                    # 8-byte rows of an MN-major A
    assert gemm(ct=_lib.BF16, ldc=12) == _lib.E_ALIGN            # 16-byte rows of C
    assert gemm(m=2 ** 20, lda=2 ** 28) == _lib.E_UNSUPPORTED     # A: 2^49 bytes
    assert gemm(la=MN, lb=MN, k=2 ** 20, lda=2 ** 28, ldb=8) == _lib.E_UNSUPPORTED  # A stored [k, m]: 2^49 bytes

    def grad(**kw):
        a = dict(dt=_lib.BF16, n=4, vocab=1000, te=4, ld_dz=1000, dz=FAKE, temp=1.0)
        a.update(kw)
        return lib.bil_linear_logp_grad(FAKE, FAKE, a["dt"], a["n"], 64, 64, a["vocab"], 64, 0, a["te"], a["temp"],
                                        FAKE, -100, FAKE, FAKE, NULL, NULL, a["dz"], a["ld_dz"], NULL)
    assert grad(dt=_lib.F32) == _lib.E_DTYPE
    assert grad(te=5) == _lib.E_INVALID_ARG
    assert grad(ld_dz=999) == _lib.E_INVALID_ARG
    assert grad(dz=NULL) == _lib.E_INVALID_ARG
    assert grad(temp=0.0) == _lib.E_INVALID_ARG
    assert grad(n=0, dz=NULL) == _lib.OK
    assert grad(n=2 ** 20, ld_dz=2 ** 28) == _lib.E_UNSUPPORTED


def test_sum_and_stream_shape_check_their_arguments(lib):
    srcs = (ctypes.c_void_p * 17)(*([0x10000] * 17))
    s = lib.bil_sum_f32
    assert s(srcs, 0, 8, FAKE, NULL) == _lib.E_INVALID_ARG          # no sources
    assert s(srcs, 17, 8, FAKE, NULL) == _lib.E_INVALID_ARG         # more than 16 sources
    assert s(srcs, 2, -1, FAKE, NULL) == _lib.E_INVALID_ARG
    assert s(srcs, 2, 8, NULL, NULL) == _lib.E_INVALID_ARG
    assert s(None, 2, 8, FAKE, NULL) == _lib.E_INVALID_ARG
    holes = (ctypes.c_void_p * 2)(0x10000, None)
    assert s(holes, 2, 8, FAKE, NULL) == _lib.E_INVALID_ARG         # a null source
    odd = (ctypes.c_void_p * 2)(0x10000, 0x10002)
    assert s(odd, 2, 8, FAKE, NULL) == _lib.E_ALIGN
    assert s(srcs, 2, 8, ctypes.c_void_p(0x10001), NULL) == _lib.E_ALIGN
    assert s(srcs, 16, 0, FAKE, NULL) == _lib.OK                    # nothing to add


    st, co, sm = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int64(0)
    shape = lib.bil_stream_shape
    assert shape(_lib.BF16, 4096, 38, 1, 0, ctypes.byref(st), ctypes.byref(co), ctypes.byref(sm)) == _lib.OK
    assert st.value >= 2 and co.value >= 1 and st.value % co.value == 0 and sm.value > 0
    assert shape(9, 4096, 38, 1, 0, ctypes.byref(st), ctypes.byref(co), ctypes.byref(sm)) == _lib.E_DTYPE
    assert shape(_lib.BF16, 12, 38, 1, 0, ctypes.byref(st), ctypes.byref(co), ctypes.byref(sm)) == \
        _lib.E_INVALID_ARG
    assert shape(_lib.BF16, 4096, 0, 1, 0, ctypes.byref(st), ctypes.byref(co), ctypes.byref(sm)) == \
        _lib.E_INVALID_ARG
    assert shape(_lib.F32, 32768, 38, 1, 0, ctypes.byref(st), ctypes.byref(co), ctypes.byref(sm)) == \
        _lib.E_UNSUPPORTED
    assert shape(_lib.BF16, 4096, 38, 1, 0, None, ctypes.byref(co), ctypes.byref(sm)) == _lib.E_INVALID_ARG
