"""The C ABI library loads, exports every function include/pa.h declares, and rejects
bad arguments on the host (none of these calls reaches the GPU)."""

import ctypes
import os
import re

import pytest

from paged_kv_decode_metadata_gb300 import binding as B
from paged_kv_decode_metadata_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_path_calls():
    names = declared_functions()
    for required in ("pa_build_metadata", "pa_decode_splitk", "pa_reduce", "pa_decode_step"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


FAKE = 1 << 20   # an aligned, never-dereferenced device address


def _splitk(lib, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, kv=0, pt=FAKE, pts=16, cl=FAKE, bs=2,
                hq=32, hkv=8, d=128, P=64, pages=100, msp=16, S=4, scale=0.1, m=FAKE, l=FAKE,
                acc=FAKE)
    args.update(over)
    a = args
    return lib.pa_decode_splitk(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["kv"], a["pt"], a["pts"],
                                a["cl"], a["bs"], a["hq"], a["hkv"], a["d"], a["P"], a["pages"],
                                a["msp"], a["S"], a["scale"], a["m"], a["l"], a["acc"], None, 1)


def test_splitk_host_validation(lib):
    assert _splitk(lib, bs=0) == B.PA_OK                      # empty batch: nothing launched
    assert _splitk(lib, q=None) == B.PA_ERR_INVALID
    assert _splitk(lib, hq=30) == B.PA_ERR_INVALID            # not a multiple of Hkv
    assert _splitk(lib, S=0) == B.PA_ERR_INVALID
    assert _splitk(lib, pts=8) == B.PA_ERR_INVALID            # stride narrower than the table
    assert _splitk(lib, q=FAKE + 8) == B.PA_ERR_INVALID       # misaligned
    assert _splitk(lib, kv=1) == B.PA_ERR_INVALID             # int8 without scales
    assert _splitk(lib, d=64) == B.PA_ERR_UNSUPPORTED
    assert _splitk(lib, P=48) == B.PA_ERR_UNSUPPORTED
    assert _splitk(lib, hq=256) == B.PA_ERR_UNSUPPORTED       # group 32
    with B.producer(B.PA_PRODUCER_FMA):
        assert _splitk(lib, hq=128) == B.PA_ERR_UNSUPPORTED   # group 16: tensor-core only


def _window(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, kv=0, pt=FAKE, pts=16, cl=FAKE, cq=None,
             bs=2, mql=1, hq=32, hkv=8, d=128, P=64, pages=100, msp=16, W=100, S=4, scale=0.1,
             m=FAKE, l=FAKE, acc=FAKE)
    a.update(over)
    return lib.pa_decode_splitk_window(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["kv"], a["pt"],
                                       a["pts"], a["cl"], a["cq"], a["bs"], a["mql"], a["hq"],
                                       a["hkv"], a["d"], a["P"], a["pages"], a["msp"], a["W"],
                                       a["S"], a["scale"], a["m"], a["l"], a["acc"], None, 1)


def test_window_host_validation(lib):
    assert _window(lib, bs=0) == B.PA_OK
    assert _window(lib, W=0) == B.PA_ERR_INVALID
    assert _window(lib, W=-3) == B.PA_ERR_INVALID
    assert _window(lib, q=None) == B.PA_ERR_INVALID
    assert _window(lib, msp=1 << 24, pts=1 << 24) == B.PA_ERR_UNSUPPORTED  # positions > 2^29
    assert _window(lib, cq=FAKE, mql=0) == B.PA_ERR_INVALID
    assert _window(lib, cq=FAKE, mql=3, hq=64) == B.PA_ERR_UNSUPPORTED       # 8 heads x 3 > 16
    with B.producer(B.PA_PRODUCER_FMA):
        assert _window(lib) == B.PA_ERR_UNSUPPORTED                       # tensor-core only
    step = lambda **o: lib.pa_decode_step_window(
        FAKE, FAKE, FAKE, 4, 1024, o.get("map", FAKE), 100, 0, 16, FAKE, FAKE, FAKE, 16,
        o.get("swa", FAKE), 16, FAKE, FAKE, FAKE, None, None, 0, 2, 32, 8, 128, 64, 100,
        o.get("W", 100), 4, 0.1, FAKE, 1 << 20, FAKE, None, None, 1)
    assert step(W=0) == B.PA_ERR_INVALID
    assert step(map=None, swa=None) == B.PA_ERR_INVALID                   # needs the SWA table


def test_host_step_validation(lib):
    base = [FAKE, FAKE, FAKE, 4, 1024, None, 0, 0, 16, FAKE, FAKE, FAKE, 16, None, 16, FAKE, FAKE,
            FAKE, None, None, 0, 2, 32, 8, 128, 64, 100, 4, 0.1, FAKE, 1 << 20, FAKE, FAKE, None, 1]
    host = lambda hq=FAKE, hr=FAKE, hs=FAKE, ho=FAKE, hl=FAKE: lib.pa_decode_step_host(
        hq, hr, hs, ho, hl, *base)
    assert host(hq=None) == B.PA_ERR_INVALID
    assert host(hr=None) == B.PA_ERR_INVALID
    assert host(ho=None) == B.PA_ERR_INVALID
    assert host(hl=None) == B.PA_ERR_INVALID                  # lse given, h_lse missing
    empty = list(base)
    empty[21] = 0                                             # bs = 0: nothing enqueued
    assert lib.pa_decode_step_host(None, None, None, None, None, *empty) == B.PA_OK


def test_packed_host_step_validation(lib):
    # pa_decode_step's arguments without the q / index / output pointers
    rest = [FAKE, 4, 1024, None, 0, 0, 16, FAKE, FAKE, FAKE, 16, None, 16, FAKE, FAKE, None,
            None, 0, 2, 32, 8, 128, 64, 100, 4, 0.1, FAKE, 1 << 20, None, 1]
    step = lambda hi=FAKE, di=FAKE, ho=FAKE, do=FAKE, bs=2: lib.pa_decode_step_host_packed(
        hi, di, ho, do, *rest[:18], bs, *rest[19:])
    assert step(hi=None) == B.PA_ERR_INVALID
    assert step(do=None) == B.PA_ERR_INVALID
    assert step(di=FAKE + 8) == B.PA_ERR_INVALID              # device buffers 16-byte aligned
    assert step(bs=0, hi=None, di=None, ho=None, do=None) == B.PA_OK
    # q bf16 then two int64 index vectors; out bf16 then lse fp32
    assert lib.pa_packed_input_bytes(3, 32, 128) == 3 * 32 * 128 * 2 + 2 * 8 * 3
    assert lib.pa_packed_output_bytes(3, 32, 128) == 3 * 32 * 128 * 2 + 4 * 3 * 32
    assert lib.pa_packed_input_bytes(0, 32, 128) == 0


def test_step_rejects_producer_limits_before_any_launch(lib):
    """A decode step the selected producer cannot run is rejected on the host before the
    metadata kernel is enqueued (here, with no GPU, an enqueue would fail as a CUDA
    error instead)."""
    step = lambda hq: lib.pa_decode_step(
        FAKE, FAKE, FAKE, 4, 1024, None, 0, 0, 16, FAKE, FAKE, FAKE, 16, None, 16, FAKE, FAKE,
        FAKE, None, None, 0, 2, hq, 2, 128, 64, 100, 4, 0.1, FAKE, 1 << 20, FAKE, None, None, 1)
    with B.producer(B.PA_PRODUCER_FMA):
        assert step(32) == B.PA_ERR_UNSUPPORTED                # CUDA-core producer: G <= 8
    window = lambda **o: lib.pa_decode_step_window(
        FAKE, FAKE, FAKE, 4, 1 << 31, FAKE, 100, 0, o.get("msp", 16), FAKE, FAKE, FAKE,
        o.get("msp", 16), FAKE, o.get("msp", 16), FAKE, FAKE, FAKE, None, None, 0, 2, 32, 8,
        128, 64, 100, 100, 4, 0.1, FAKE, 1 << 20, FAKE, None, None, 1)
    assert window(msp=(1 << 23) + 1) == B.PA_ERR_UNSUPPORTED   # window bounds past 2^29
    with B.producer(B.PA_PRODUCER_FMA):
        assert window() == B.PA_ERR_UNSUPPORTED                # tensor-core producer only


def test_multi_step_validation(lib):
    def step(cq=FAKE, mql=2, hq=32, bs=2, total_q=4):
        return lib.pa_decode_step_multi(
            FAKE, FAKE, FAKE, 4, 1024, None, 0, 0, 16, FAKE, FAKE, FAKE, 16, None, 16, FAKE,
            B.PA_Q_MODE_CUMSUM, 0, cq, FAKE, total_q, mql, FAKE, FAKE, None, None, 0, bs, hq, 8,
            128, 64, 100, 4, 0.1, FAKE, 1 << 30, FAKE, None, None, 1)
    assert step(bs=0) == B.PA_OK
    assert step(cq=None) == B.PA_ERR_INVALID
    assert step(mql=0) == B.PA_ERR_INVALID
    assert step(hq=30) == B.PA_ERR_INVALID
    assert step(hq=64, mql=3) == B.PA_ERR_UNSUPPORTED       # 8 heads x 3 queries > 16
    with B.producer(B.PA_PRODUCER_FMA):
        assert step() == B.PA_ERR_UNSUPPORTED


def test_window_pages():
    # the most pages W + max_q_len - 1 consecutive positions can touch, capped
    assert B.pa_window_pages(4096, 1, 64, 256) == 65
    assert B.pa_window_pages(4096, 1, 64, 40) == 40
    assert B.pa_window_pages(6, 3, 4, 4) == 3
    assert B.pa_window_pages(8, 3, 4, 4) == 4
    assert B.pa_window_pages(1, 1, 16, 100) == 2
    assert B.pa_window_pages(64, 1, 64, 100) == 2
    assert B.pa_window_pages(0, 1, 64, 100) == 0
    assert B.pa_window_pages(10, 0, 64, 100) == 0


def test_producer_selection(lib):
    prev = B.pa_select_producer(B.PA_PRODUCER_FMA)
    assert B.pa_select_producer(B.PA_PRODUCER_MMA) == B.PA_PRODUCER_FMA
    assert B.pa_select_producer(7) == B.PA_PRODUCER_MMA          # unknown: no change
    assert B.pa_select_producer(prev) == B.PA_PRODUCER_MMA


def test_reduce_and_metadata_host_validation(lib):
    assert lib.pa_reduce(FAKE, FAKE, FAKE, 0, 32, 128, 4, FAKE, None, None, 1) == B.PA_OK
    assert lib.pa_reduce(None, FAKE, FAKE, 1, 32, 128, 4, FAKE, None, None, 1) == B.PA_ERR_INVALID
    assert lib.pa_reduce(FAKE, FAKE, FAKE, 1, 32, 64, 4, FAKE, None, None, 1) == B.PA_ERR_UNSUPPORTED
    md = lambda **o: lib.pa_build_metadata(
        o.get("rpi", FAKE), FAKE, FAKE, 4, o.get("r2ts", 1024), o.get("map", None), 0, FAKE, FAKE,
        FAKE, o.get("pts", 16), o.get("swa", None), 16, o.get("bs", 2), 0, 16, 64, None, 1)
    assert md(bs=0) == B.PA_OK
    assert md(rpi=None) == B.PA_ERR_INVALID
    assert md(r2ts=15 * 64) == B.PA_ERR_INVALID               # column 15*64 outside the row
    assert md(pts=8) == B.PA_ERR_INVALID
    assert md(map=FAKE) == B.PA_ERR_INVALID                   # mapping without swa output
    assert md(swa=FAKE) == B.PA_ERR_INVALID                   # swa output without mapping


def test_workspace_and_split_heuristic(lib):
    assert B.pa_workspace_bytes(32, 32, 128, 10) == 2 * 10240 * 4 + 10240 * 128 * 4
    assert B.pa_workspace_bytes(0, 32, 128, 4) == 0
    for kv in (B.PA_KV_BF16, B.PA_KV_INT8):
        for bs, hkv, pages in ((1, 8, 16), (8, 8, 16), (1, 8, 128), (32, 8, 128), (64, 8, 256),
                               (64, 8, 65), (1, 1, 1)):
            s = B.pa_choose_splits(bs, hkv, pages, 64, kv, 152)
            assert 1 <= s <= max(1, pages)
            pps = -(-pages // s)
            assert -(-pages // pps) == s          # the longest request has no empty split
    # the GB300 sweeps' best counts: bs32 ctx8K bf16, bs64 ctx8K int8, bs64 ctx16K int8
    # (6 and 8 equal), bs64 window 4096 int8
    assert B.pa_choose_splits(32, 8, 128, 64, B.PA_KV_BF16, 152) == 5
    assert B.pa_choose_splits(64, 8, 128, 64, B.PA_KV_INT8, 152) == 4
    assert B.pa_choose_splits(64, 8, 256, 64, B.PA_KV_INT8, 152) == 8
    assert B.pa_choose_splits(64, 8, 65, 64, B.PA_KV_INT8, 152) == 3
    assert B.pa_choose_splits(0, 8, 16, 64, B.PA_KV_BF16, 152) == 1
    assert B.pa_status_string(B.PA_ERR_UNSUPPORTED) == "unsupported shape"


TS_HEADER = os.path.join(os.path.dirname(HEADER), "pa_timestamps.h")


def test_instrumented_build_exports_its_header_and_production_does_not():
    build.build(instrumented=True)
    ts = B.load_instrumented()
    text = re.sub(r"/\*.*?\*/", "", open(TS_HEADER).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))
    assert names == ["pa_set_test_hold_loads", "pa_set_test_no_persist", "pa_set_timestamp_buffer"]
    for n in names + declared_functions():
        assert hasattr(ts, n), n
    prod = ctypes.CDLL(build.LIB_PATH)
    for n in names:
        assert not hasattr(prod, n), n


def _exported(path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return sorted(line.split()[-1] for line in out.splitlines() if line.strip())


def test_library_exports_exactly_the_c_abi(lib):
    assert _exported(build.LIB_PATH) == declared_functions()
