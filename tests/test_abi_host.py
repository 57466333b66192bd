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


def test_contract_id_and_status_strings(lib):
    cid = _lib.contract_id()
    assert cid.startswith("bil.v3") and "ex2.approx" in cid and "fma" in cid and "entropy" in cid
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
