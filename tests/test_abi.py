"""The C ABI library loads and exports every declared symbol; host-side checks
work without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_112_gb300 as pkv
from paged_kv_cache_112_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    try:
        pkv_build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    return pkv.load()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["pkv_write_cache", "pkv_copy_blocks", "pkv_decode_attention", "pkv_decode_partitions",
              "pkv_decode_reduce", "pkv_decode_workspace_bytes", "pkv_status_string", "pkv_version",
              "pkv_write_cache_fp8", "pkv_copy_blocks_fp8", "pkv_decode_attention_fp8", "pkv_swap_blocks"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(pkv.library_path())
    for name in _declared():
        assert hasattr(raw, name), name


def test_status_strings_and_version(lib):
    assert pkv.status_string(pkv.PKV_OK) == "PKV_OK"
    assert pkv.status_string(pkv.PKV_ERR_WORKSPACE) == "PKV_ERR_WORKSPACE"
    assert lib.pkv_version() >= 100


def test_workspace_bytes(lib):
    # no split -> nothing needed
    assert pkv.decode_workspace_bytes(64, 32, 128, 2048, 0) == 0
    assert pkv.decode_workspace_bytes(64, 32, 128, 512, 512) == 0
    # 8 seqs x 32 heads x 256 partitions: acc fp32 [.., 128] + (m, l) pairs, each 256-B aligned,
    # then the 256-byte control block of the work queue
    rows = 8 * 32 * 256
    acc = rows * 128 * 4
    ml = rows * 8
    up = lambda x: (x + 255) // 256 * 256
    assert pkv.decode_workspace_bytes(8, 32, 128, 131072, 512) == up(acc) + up(ml)
    assert pkv.decode_workspace_bytes(8, 32, 128, 100, 24) == 0  # not a multiple of 16 -> invalid
    # balanced split: per-pair metadata + 2 partial records per warp (group <= 8 heads); without a
    # device the SM count defaults to 256, else the device's
    bal = pkv.decode_workspace_bytes(64, 32, 128, 2048, pkv.PARTITION_BALANCED)
    assert bal >= 64 * 32 * 8 + 256 * 0  # at least the metadata
    assert pkv.decode_workspace_bytes(64, 32, 128, 2048, -2) == 0


FAKE = 0x10000  # never dereferenced: validation fails before any device work


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bs=0, bt=FAKE, maxb=4, cl=FAKE, S=2, Hq=8, Hkv=2, D=128, B=16, NB=10,
             scale=0.1, ps=0, maxlen=64, ws=None, wsb=0, kvd=pkv.PKV_BF16, od=pkv.PKV_F32)
    a.update(kw)
    return lib.pkv_decode_attention(a["out"], a["q"], a["k"], a["v"], a["bs"], a["bt"], a["maxb"], a["cl"], a["S"],
                                    a["Hq"],
                                    a["Hkv"], a["D"], a["B"], a["NB"], a["scale"], a["ps"], a["maxlen"], a["ws"],
                                    a["wsb"], a["kvd"], a["od"], None, None)


def test_decode_argument_validation(lib):
    assert _decode(lib, B=24) == pkv.PKV_ERR_UNSUPPORTED  # block sizes: 8, 16, 32, 64
    assert _decode(lib, B=128) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(lib, B=32, ps=pkv.PARTITION_BALANCED) == pkv.PKV_ERR_UNSUPPORTED  # balanced split: 16 only
    assert _decode(lib, D=96) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(lib, Hq=6, Hkv=4) == pkv.PKV_ERR_UNSUPPORTED  # not a whole group
    assert _decode(lib, Hq=32, Hkv=2) == pkv.PKV_ERR_UNSUPPORTED  # group 16 > 8
    assert _decode(lib, ps=24) == pkv.PKV_ERR_UNSUPPORTED
    assert _decode(lib, q=None) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(lib, k=FAKE + 8) == pkv.PKV_ERR_INVALID_ARG  # pool not 16-byte aligned
    assert _decode(lib, kvd=pkv.PKV_F32) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(lib, S=-1) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(lib, scale=float("nan")) == pkv.PKV_ERR_INVALID_ARG
    # block stride: below a dense block, or not a whole 16-byte vector
    assert _decode(lib, bs=16 * 2 * 128 - 8) == pkv.PKV_ERR_INVALID_ARG
    assert _decode(lib, bs=3 * 16 * 2 * 128 + 4) == pkv.PKV_ERR_INVALID_ARG
    # split needs a workspace
    assert _decode(lib, ps=16, maxlen=64) == pkv.PKV_ERR_WORKSPACE
    need = pkv.decode_workspace_bytes(2, 8, 128, 64, 16)
    assert _decode(lib, ps=16, maxlen=64, ws=FAKE, wsb=need - 1) == pkv.PKV_ERR_WORKSPACE


def test_write_and_copy_argument_validation(lib):
    w = lambda **kw: lib.pkv_write_cache(kw.get("kn", FAKE), kw.get("vn", FAKE), FAKE, FAKE, kw.get("bs", 0), FAKE,
                                         kw.get("T", 4), kw.get("stride", 0), kw.get("Hkv", 8), kw.get("D", 128),
                                         kw.get("B", 16), 100, kw.get("dt", pkv.PKV_F16), None, None)
    assert w(B=12) == pkv.PKV_ERR_UNSUPPORTED
    assert w(T=-1) == pkv.PKV_ERR_INVALID_ARG
    assert w(kn=None) == pkv.PKV_ERR_INVALID_ARG
    assert w(kn=FAKE + 2) == pkv.PKV_ERR_INVALID_ARG  # rows must be 16-byte aligned
    assert w(stride=100) == pkv.PKV_ERR_INVALID_ARG  # stride below a row
    assert w(Hkv=1, D=4) == pkv.PKV_ERR_UNSUPPORTED  # row not a whole 16-byte vector
    assert w(T=0) == pkv.PKV_OK  # no-op, no launch
    assert w(bs=16 * 8 * 128 - 8) == pkv.PKV_ERR_INVALID_ARG  # block stride below a dense block
    c = lambda **kw: lib.pkv_copy_blocks(FAKE, FAKE, kw.get("pairs", FAKE), kw.get("P", 3), kw.get("layers", 1), 8,
                                         128, kw.get("B", 16), 100, pkv.PKV_BF16, None, None)
    assert c(B=12) == pkv.PKV_ERR_UNSUPPORTED
    assert c(layers=0) == pkv.PKV_ERR_INVALID_ARG
    assert c(pairs=None) == pkv.PKV_ERR_INVALID_ARG
    assert c(P=0) == pkv.PKV_OK


def test_fp8_argument_validation(lib):
    def d(**kw):
        a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, bt=FAKE, maxb=4, cl=FAKE, S=2, Hq=8, Hkv=2,
                 D=128, B=16, NB=10, L=1, scale=0.1, ps=0, maxlen=64, ws=None, wsb=0, qd=pkv.PKV_BF16,
                 od=pkv.PKV_F32)
        a.update(kw)
        return lib.pkv_decode_attention_fp8(a["out"], a["q"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["maxb"],
                                            a["cl"], a["S"], a["Hq"], a["Hkv"], a["D"], a["B"], a["NB"], a["L"],
                                            a["scale"], a["ps"], a["maxlen"], a["ws"], a["wsb"], a["qd"], a["od"],
                                            None, None)

    assert d(D=64) == pkv.PKV_ERR_UNSUPPORTED  # FP8 tiles: head_dim 128 only
    # balanced split: needs its workspace (no device here: the SM-count query fails first)
    assert d(ps=pkv.PARTITION_BALANCED) in (pkv.PKV_ERR_WORKSPACE, pkv.PKV_ERR_CUDA)
    assert d(B=8) == pkv.PKV_ERR_UNSUPPORTED
    assert d(ks=None) == pkv.PKV_ERR_INVALID_ARG
    assert d(vs=FAKE + 2) == pkv.PKV_ERR_INVALID_ARG
    assert d(q=FAKE + 8) == pkv.PKV_ERR_INVALID_ARG  # q rows are read as 16-byte vectors
    assert d(qd=pkv.PKV_F32) == pkv.PKV_ERR_INVALID_ARG
    assert d(ps=16, maxlen=64) == pkv.PKV_ERR_WORKSPACE
    # the fused FP8 step needs fixed partitions (the balanced split has no fused write)
    assert lib.pkv_decode_step_fp8(FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 8, 2,
                                   128, 16, 10, 1, 0.1, pkv.PARTITION_BALANCED, 64, None, 0, pkv.PKV_BF16,
                                   pkv.PKV_F32, None, None) == pkv.PKV_ERR_UNSUPPORTED
    assert d(L=0) == pkv.PKV_ERR_INVALID_ARG  # layers per block: 1..4096
    assert d(L=4097) == pkv.PKV_ERR_INVALID_ARG
    assert d(S=0) == pkv.PKV_OK
    assert d(S=0, L=32) == pkv.PKV_OK
    w = lambda **kw: lib.pkv_write_cache_fp8(FAKE, FAKE, FAKE, FAKE, kw.get("ks", FAKE), FAKE, FAKE, kw.get("T", 4),
                                             kw.get("stride", 0), 8, kw.get("D", 128), kw.get("B", 16), 100,
                                             kw.get("L", 1), kw.get("dt", pkv.PKV_BF16), None, None)
    assert w(D=72) == pkv.PKV_ERR_UNSUPPORTED  # 16 codes per vector within one head
    assert w(B=32) == pkv.PKV_ERR_UNSUPPORTED
    assert w(ks=None) == pkv.PKV_ERR_INVALID_ARG
    assert w(dt=pkv.PKV_F32) == pkv.PKV_ERR_INVALID_ARG
    assert w(stride=12) == pkv.PKV_ERR_INVALID_ARG
    assert w(L=0) == pkv.PKV_ERR_INVALID_ARG
    assert w(T=0) == pkv.PKV_OK
    c = lambda **kw: lib.pkv_copy_blocks_fp8(FAKE, FAKE, kw.get("ks", FAKE), FAKE, FAKE, kw.get("P", 3),
                                             kw.get("L", 1), 8, 128, kw.get("B", 16), 100, None, None)
    assert c(B=8) == pkv.PKV_ERR_UNSUPPORTED
    assert c(L=0) == pkv.PKV_ERR_INVALID_ARG
    assert c(ks=None) == pkv.PKV_ERR_INVALID_ARG
    assert c(P=0) == pkv.PKV_OK


def test_swap_argument_validation(lib):
    def sw(**kw):
        return lib.pkv_swap_blocks(kw.get("dk", FAKE), FAKE, kw.get("ds", 4096), 10, FAKE, FAKE, kw.get("ss", 4096), 10,
                                   kw.get("bb", 4096), kw.get("pairs", FAKE), kw.get("P", 3), None, None)

    assert sw(bb=4000) == pkv.PKV_ERR_INVALID_ARG  # not a whole 16-byte vector
    assert sw(ds=2048) == pkv.PKV_ERR_INVALID_ARG  # stride below a block
    assert sw(ss=4104) == pkv.PKV_ERR_INVALID_ARG  # stride not a 16-byte multiple
    assert sw(dk=FAKE + 8) == pkv.PKV_ERR_INVALID_ARG
    assert sw(pairs=None) == pkv.PKV_ERR_INVALID_ARG
    assert sw(P=-1) == pkv.PKV_ERR_INVALID_ARG
    assert sw(P=0) == pkv.PKV_OK
    # pointers the device cannot reach (here: no device at all, or plain host memory) are refused
    host = ctypes.create_string_buffer(8192 + 16)
    addr = (ctypes.addressof(host) + 15) // 16 * 16
    assert sw(dk=addr) == pkv.PKV_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from paged_kv_cache_112_gb300 import _binding

    monkeypatch.setattr(_binding, "_LIB", None)
    monkeypatch.setattr(_binding._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(pkv.PkvError):
        _binding.load()


def test_bounded_wait_check_argument_validation(lib):
    """Rejected before any launch: negative or over-long limits, a missing or
    misaligned status word."""
    fake = 256
    assert lib.pkv_check_bounded_wait(-1, 0, fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_check_bounded_wait(2_000_000_001, 0, fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_check_bounded_wait(1000, 0, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_check_bounded_wait(1000, 0, fake + 2, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_check_bounded_wait(1000, 2, fake, None) == pkv.PKV_ERR_INVALID_ARG
