"""The C ABI on the host: the library builds, loads without a GPU, exports every
function include/pskv.h declares, and its host-only entry points (sizes, the
byte contract, refusals made before any launch) behave as documented."""
import ctypes
import json
import os
import re

import pytest

import paged_split_kv_attn_gb300 as pskv
from paged_split_kv_attn_gb300 import _binding as B
from paged_split_kv_attn_gb300 import build as pskv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pskv.h")


@pytest.fixture(scope="module")
def lib():
    pskv_build.build()
    return pskv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return [n for n in names if not n.startswith("__")]


def test_header_declarations_match_the_binding():
    assert sorted(declared_functions()) == sorted(B.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_strerror(lib):
    assert pskv.pskv_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert pskv.pskv_strerror(code) != "unknown status"
    assert pskv.pskv_strerror(-99) == "unknown status"


def test_partial_scratch_contract_matches_the_page(lib):
    with open(os.path.join(ROOT, "tests", "golden", "gem_scratch_contract.json")) as f:
        g = json.load(f)
    s = g["shape"]
    for c in g["cases"]:
        got = pskv.pskv_partial_scratch_bytes(s["batch"], s["num_q_heads"], s["head_dim_v"],
                                              c["num_splits"])
        assert got == (c["maxima"], c["denominators"], c["numerators"], c["total"])
    for p, mib in g["numerator_mib_by_splits"].items():
        assert pskv.pskv_partial_scratch_bytes(1, 32, 512, int(p))[2] == mib << 20


def test_size_overflow_fails_closed(lib):
    with pytest.raises(pskv.PskvError) as e:
        pskv.pskv_partial_scratch_bytes(1 << 40, 1 << 20, 512, 1 << 10)
    assert e.value.code == B.PSKV_ERR_OVERFLOW
    with pytest.raises(pskv.PskvError) as e:
        pskv.decode_attn_workspace_bytes(1 << 30, 1 << 30, 512, 1024)
    assert e.value.code == B.PSKV_ERR_OVERFLOW
    with pytest.raises(pskv.PskvError):
        pskv.decode_attn_workspace_bytes(1, 32, 512, PSKV_MAX + 1)


PSKV_MAX = B.PSKV_MAX_SPLITS


def test_workspace_holds_the_partials(lib):
    """The decode workspace is the partial buffer (256-byte aligned sections);
    the merge keeps its group states on chip."""
    for p in (1, 16, 17, 32, 256, 1024):
        n = pskv.decode_attn_workspace_bytes(2, 32, 512, p)
        partial = pskv.pskv_partial_scratch_bytes(2, 32, 512, p)[3]
        assert partial <= n <= partial + 3 * 256
        assert n % 256 == 0
        assert pskv.merge_partials_workspace_bytes(64, p, 512) == 0
    assert pskv.decode_attn_workspace_bytes(1, 32, 512, 0) == \
        pskv.decode_attn_workspace_bytes(1, 32, 512, B.PSKV_AUTO_MAX_SPLITS)


def _desc(**kw):
    base = dict(num_pages=8, page_size=256, num_kv_heads=4, head_dim_k=512, head_dim_v=512,
                kv_dtype=B.PSKV_DTYPE_BF16, format=B.PSKV_FORMAT_SPLIT, k_pool=0x10000,
                v_pool=0x20000, status=None)
    base.update(kw)
    return B.LayoutDesc(*[base[f] for f, _ in B.LayoutDesc._fields_])


@pytest.mark.parametrize("kw,code", [
    (dict(), 0),
    (dict(head_dim_k=256, head_dim_v=256, page_size=64), 0),
    (dict(kv_dtype=B.PSKV_DTYPE_F32), 0),
    (dict(k_pool=None), B.PSKV_ERR_INVALID_ARG),
    (dict(v_pool=0x20008), B.PSKV_ERR_INVALID_ARG),       # not 16-byte aligned
    (dict(page_size=100), B.PSKV_ERR_INVALID_ARG),        # not a multiple of the key tile
    (dict(num_pages=0), B.PSKV_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), B.PSKV_ERR_INVALID_ARG),
    (dict(kv_dtype=7), B.PSKV_ERR_INVALID_ARG),
    (dict(format=B.PSKV_FORMAT_FOLDED), B.PSKV_ERR_UNSUPPORTED),
    (dict(head_dim_k=128, head_dim_v=128), B.PSKV_ERR_UNSUPPORTED),
    (dict(head_dim_v=256), B.PSKV_ERR_UNSUPPORTED),
])
def test_layout_validation(lib, kw, code):
    d = _desc(**kw)
    h = ctypes.c_void_p()
    rc = lib.paged_kv_layout_create(ctypes.byref(d), ctypes.byref(h))
    assert rc == code
    if rc == 0:
        assert h.value
        lib.paged_kv_layout_destroy(h)
    else:
        assert not h.value


def _layout(lib, **kw):
    d = _desc(**kw)
    h = ctypes.c_void_p()
    assert lib.paged_kv_layout_create(ctypes.byref(d), ctypes.byref(h)) == 0
    return h


def _decode_rc(lib, layout, lens, **kw):
    args = dict(q=0x30000, tables=0x40000, stride=4, lens_dev=0x50000, batch=len(lens), hq=32,
                scale=0.04, splits=8, ws=0x60000, ws_bytes=1 << 30, out=0x70000,
                out_dtype=B.PSKV_DTYPE_BF16)
    args.update(kw)
    lh = (ctypes.c_int32 * len(lens))(*lens)
    return lib.decode_attn_splitkv(layout, args["q"], args["tables"], args["stride"], lh,
                                   args["lens_dev"], args["batch"], args["hq"], args["scale"],
                                   args["splits"], args["ws"], args["ws_bytes"], args["out"],
                                   args["out_dtype"], None, None)


def test_decode_refusals_happen_before_any_launch(lib):
    """Every refusal below is decided on the host, so it runs without a GPU."""
    h = _layout(lib)
    try:
        assert _decode_rc(lib, h, [100], q=None) == B.PSKV_ERR_INVALID_ARG
        assert _decode_rc(lib, h, [0]) == B.PSKV_ERR_INVALID_ARG           # empty row
        assert _decode_rc(lib, h, [4 * 256 + 1]) == B.PSKV_ERR_INVALID_ARG  # past the table
        assert _decode_rc(lib, h, [100], hq=30) == B.PSKV_ERR_UNSUPPORTED  # 30 % 4 != 0
        assert _decode_rc(lib, h, [100], hq=4 * 16) == B.PSKV_ERR_UNSUPPORTED  # G = 16 at D = 512
        assert _decode_rc(lib, h, [100], splits=-1) == B.PSKV_ERR_INVALID_ARG
        assert _decode_rc(lib, h, [100], splits=PSKV_MAX + 1) == B.PSKV_ERR_INVALID_ARG
        assert _decode_rc(lib, h, [100], scale=float("nan")) == B.PSKV_ERR_INVALID_ARG
        assert _decode_rc(lib, h, [100], out_dtype=5) == B.PSKV_ERR_INVALID_ARG
        assert _decode_rc(lib, h, [100], q=0x30008) == B.PSKV_ERR_INVALID_ARG  # misaligned
        assert _decode_rc(lib, h, [100], ws_bytes=1024) == B.PSKV_ERR_WORKSPACE_TOO_SMALL
    finally:
        lib.paged_kv_layout_destroy(h)


def _multirow_rc(lib, layout, lens, tokens, **kw):
    args = dict(q=0x30000, tables=0x40000, stride=4, lens_dev=0x50000, batch=len(lens), hq=32,
                scale=0.04, splits=8, ws=0x60000, ws_bytes=1 << 30, out=0x70000,
                out_dtype=B.PSKV_DTYPE_BF16)
    args.update(kw)
    lh = (ctypes.c_int32 * len(lens))(*lens)
    return lib.decode_attn_multirow(layout, args["q"], args["tables"], args["stride"], lh,
                                    args["lens_dev"], args["batch"], tokens, args["hq"],
                                    args["scale"], args["splits"], args["ws"], args["ws_bytes"],
                                    args["out"], args["out_dtype"], None, None)


def test_multirow_refusals_happen_before_any_launch(lib):
    h = _layout(lib)
    f32 = _layout(lib, kv_dtype=B.PSKV_DTYPE_F32)
    try:
        assert _multirow_rc(lib, h, [100], 0) == B.PSKV_ERR_INVALID_ARG
        assert _multirow_rc(lib, h, [100], B.PSKV_MAX_WINDOW_TOKENS + 1) == B.PSKV_ERR_INVALID_ARG
        assert _multirow_rc(lib, h, [3], 4) == B.PSKV_ERR_INVALID_ARG   # row shorter than the window
        assert _multirow_rc(lib, f32, [100], 2) == B.PSKV_ERR_UNSUPPORTED  # tensor-core family only
        # the workspace holds batch x tokens rows of partials
        need = pskv.decode_attn_workspace_bytes(2, 32, 512, 8)
        assert _multirow_rc(lib, h, [100, 100], 3, ws_bytes=need) == B.PSKV_ERR_WORKSPACE_TOO_SMALL
    finally:
        lib.paged_kv_layout_destroy(h)
        lib.paged_kv_layout_destroy(f32)


def _prep_rc(lib, layout, rot=128, stride=40 * 512, cols=(0, 32 * 512, 36 * 512), w_k=0x90000,
             host=None, n=1):
    desc = B.PrepDesc(rot_dims=rot, eps=1e-6, w_q=0x80000, w_k=w_k, rope_cos=0xa0000,
                      rope_sin=0xb0000, max_pos=4096)
    hr = hp = hl = None
    if host is not None:
        hr, hp, hl = ((ctypes.c_int32 * len(v))(*v) for v in host)
    return lib.kv_prep_append(layout, ctypes.byref(desc), 0x10000, stride, cols[0], cols[1],
                              cols[2], n, 32, 0x20000, 0x30000, None, 0x40000, 4, 0x50000, 1,
                              hr, hp, hl, 0x60000, None)


def test_prep_refusals_happen_before_any_launch(lib):
    h = _layout(lib)
    f32 = _layout(lib, kv_dtype=B.PSKV_DTYPE_F32)
    folded = _layout(lib, format=B.PSKV_FORMAT_FOLDED, head_dim_k=128)
    try:
        assert _prep_rc(lib, f32) == B.PSKV_ERR_UNSUPPORTED             # bf16 pools only
        assert _prep_rc(lib, h, rot=127) == B.PSKV_ERR_INVALID_ARG      # odd rotation
        assert _prep_rc(lib, h, rot=514) == B.PSKV_ERR_INVALID_ARG      # wider than the head
        assert _prep_rc(lib, h, stride=39 * 512) == B.PSKV_ERR_INVALID_ARG  # V band past the row
        assert _prep_rc(lib, h, cols=(4, 32 * 512, 36 * 512)) == B.PSKV_ERR_INVALID_ARG
        assert _prep_rc(lib, h, host=([0], [4 * 256], [4])) == B.PSKV_ERR_PAST_PAGES
        # folded: K and V from one band, K's multiplier given, the rotated quarter stored
        assert _prep_rc(lib, folded) == B.PSKV_ERR_UNSUPPORTED
        assert _prep_rc(lib, folded, cols=(0, 32 * 512, 32 * 512), w_k=None) == \
            B.PSKV_ERR_UNSUPPORTED
        assert _prep_rc(lib, folded, rot=64, cols=(0, 32 * 512, 32 * 512)) == \
            B.PSKV_ERR_UNSUPPORTED
        assert _prep_rc(lib, h, n=0) == 0                                # nothing to do
    finally:
        for x in (h, f32, folded):
            lib.paged_kv_layout_destroy(x)


def _prefill_rc(lib, layout, lens, cu, window=0, splits=1, ws_bytes=0, hq=32):
    lh = (ctypes.c_int32 * len(lens))(*lens)
    ch = (ctypes.c_int32 * len(cu))(*cu)
    return lib.prefill_attn_paged(layout, 0x30000, ch, 0x38000, 0x40000, 4, lh, 0x50000,
                                  len(lens), hq, window, 0.04, splits,
                                  0x60000 if ws_bytes else None, ws_bytes, 0x70000,
                                  B.PSKV_DTYPE_BF16, None, None)


def test_prefill_refusals_happen_before_any_launch(lib):
    h = _layout(lib)
    f32 = _layout(lib, kv_dtype=B.PSKV_DTYPE_F32)
    try:
        assert _prefill_rc(lib, h, [100, 50], [1, 5, 9]) == B.PSKV_ERR_INVALID_ARG  # not from 0
        assert _prefill_rc(lib, h, [100, 50], [0, 5, 2]) == B.PSKV_ERR_INVALID_ARG  # decreasing
        assert _prefill_rc(lib, h, [100, 50], [0, 5, 56]) == B.PSKV_ERR_INVALID_ARG  # 51 > 50 keys
        assert _prefill_rc(lib, h, [100, 50], [0, 0, 0]) == B.PSKV_ERR_INVALID_ARG  # no token
        assert _prefill_rc(lib, h, [100], [0, 5], window=-1) == B.PSKV_ERR_INVALID_ARG
        assert _prefill_rc(lib, f32, [100], [0, 5]) == B.PSKV_ERR_UNSUPPORTED  # tensor-core only
        # query heads per KV head: a power of two up to 128 (a block of 128 columns)
        assert _prefill_rc(lib, h, [100], [0, 5], hq=12) == B.PSKV_ERR_UNSUPPORTED   # G = 3
        assert _prefill_rc(lib, h, [100], [0, 5], hq=1024) == B.PSKV_ERR_UNSUPPORTED  # G = 256
        # several partitions need the partial buffer
        assert _prefill_rc(lib, h, [100], [0, 5], splits=2) == B.PSKV_ERR_WORKSPACE_TOO_SMALL
    finally:
        lib.paged_kv_layout_destroy(h)
        lib.paged_kv_layout_destroy(f32)


def test_append_past_pages_refused_on_host(lib):
    h = _layout(lib)
    try:
        rows = (ctypes.c_int32 * 2)(0, 1)
        pos = (ctypes.c_int32 * 2)(10, 3 * 256)        # row 1 leases 3 pages: 768 is past them
        lease = (ctypes.c_int32 * 2)(1, 3)
        rc = lib.kv_append_rows(h, 0x10000, 0x20000, 0x30000, 0x40000, 2, 0x50000, 4, 0x60000, 2,
                                rows, pos, lease, None)
        assert rc == B.PSKV_ERR_PAST_PAGES
        # only some of the host copies: refused as an argument error
        rc = lib.kv_append_rows(h, 0x10000, 0x20000, 0x30000, 0x40000, 2, 0x50000, 4, 0x60000, 2,
                                rows, None, lease, None)
        assert rc == B.PSKV_ERR_INVALID_ARG
        assert lib.kv_append_rows(h, 0x10000, 0x20000, 0x30000, 0x40000, 0, 0x50000, 4, 0x60000,
                                  2, None, None, None, None) == 0  # nothing to do
    finally:
        lib.paged_kv_layout_destroy(h)


def test_merge_refusals(lib):
    P = ctypes.c_void_p
    assert lib.merge_partials(None, 0x10, 0x20, 4, 8, 512, 0x30, 0, None, 0, None, None,
                              None) == B.PSKV_ERR_INVALID_ARG
    assert lib.merge_partials(0x10, 0x10, 0x20, 4, 8, 510, 0x30, 0, None, 0, None, None,
                              None) == B.PSKV_ERR_INVALID_ARG  # dv not a multiple of 4
    one = B.DecodeOpts(1, None, None)  # groups of one partial: 65 groups are more than 64
    assert lib.merge_partials(0x10, 0x10, 0x20, 4, 65, 512, 0x30, 0, None, 0, None,
                              ctypes.byref(one), None) == B.PSKV_ERR_INVALID_ARG
    opts = B.DecodeOpts(17, None, None)
    assert lib.merge_partials(0x10, 0x10, 0x20, 4, 8, 512, 0x30, 0, None, 0, None,
                              ctypes.byref(opts), None) == B.PSKV_ERR_INVALID_ARG
    del P


def test_workspace_size_queries_follow_the_plan(lib):
    """With an explicit split count the planning is host-only: the size queries
    answer the bytes of the plan's partials (0 for one partition, which writes
    its output directly) and refuse what the call would refuse."""
    h = _layout(lib)
    out = ctypes.c_size_t()
    try:
        lh = (ctypes.c_int32 * 2)(900, 50)
        ch = (ctypes.c_int32 * 3)(0, 40, 70)
        for splits, rows_bytes in ((1, 0), (2, pskv.decode_attn_workspace_bytes(70, 32, 512, 2)),
                                   (5, pskv.decode_attn_workspace_bytes(70, 32, 512, 5))):
            assert lib.prefill_attn_workspace_bytes(h, ch, lh, 4, 2, 32, 0, splits,
                                                    ctypes.byref(out)) == 0
            assert out.value == rows_bytes
        bad = (ctypes.c_int32 * 3)(0, 40, 91)  # the second row: 51 tokens on 50 keys
        assert lib.prefill_attn_workspace_bytes(h, bad, lh, 4, 2, 32, 0, 2,
                                                ctypes.byref(out)) == B.PSKV_ERR_INVALID_ARG
        assert lib.prefill_attn_workspace_bytes(h, ch, lh, 4, 2, 32, 0, 2,
                                                None) == B.PSKV_ERR_INVALID_ARG
        # verify windows and drafted trees: batch x tokens rows of partials
        for tree in (0, 1):
            assert lib.decode_attn_multirow_workspace_bytes(h, lh, 4, 2, 3, 32, tree, 7,
                                                            ctypes.byref(out)) == 0
            assert out.value == pskv.decode_attn_workspace_bytes(6, 32, 512, 7)
            assert lib.decode_attn_multirow_workspace_bytes(h, lh, 4, 2, 3, 32, tree, 1,
                                                            ctypes.byref(out)) == 0
            assert out.value == 0
        assert lib.decode_attn_multirow_workspace_bytes(h, lh, 4, 2, 65, 32, 0, 7,
                                                        ctypes.byref(out)) == B.PSKV_ERR_INVALID_ARG
        assert lib.decode_attn_multirow_workspace_bytes(None, lh, 4, 2, 3, 32, 0, 7,
                                                        ctypes.byref(out)) == B.PSKV_ERR_INVALID_ARG
    finally:
        lib.paged_kv_layout_destroy(h)
