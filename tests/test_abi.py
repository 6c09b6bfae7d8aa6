"""The C ABI: the library builds for sm_103a, loads, exports every declared
entry point, and its host-side logic (budget arithmetic, argument checks that
return before any CUDA call) behaves as declared. No GPU needed."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsel.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    import attention_score_vision_gb300 as tsel
    tsel.build()
    return tsel.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsel_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("tsel_importance", "tsel_select_topk", "tsel_gather_compact",
              "tsel_importance_workspace_size", "tsel_keep_count", "tsel_read_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_no_unexpected_exports(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {n for n in exported if n.startswith("tsel_")}
    assert ours == set(_declared_functions())


@pytest.mark.parametrize("n,permille,text,total", [(3072, 300, 142, 1063), (896, 800, 142, 858),
                                                   (3072, 700, 142, 2292), (896, 900, 142, 948)])
def test_keep_count_matches_the_pages(lib, n, permille, text, total):
    assert lib.tsel_keep_count(n, permille) + text == total


def test_keep_count_edges(lib):
    import attention_score_vision_gb300 as tsel
    assert tsel.tsel_keep_count(0, 600) == 0
    assert tsel.tsel_keep_count(16384, 1000) == 16384
    assert tsel.tsel_keep_count(2**31 - 1, 999) == (2**31 - 1) * 999 // 1000
    assert tsel.tsel_keep_count(-1, 500) == -1


def test_status_strings(lib):
    import attention_score_vision_gb300 as tsel
    assert tsel.tsel_status_string(0) == "TSEL_OK"
    assert tsel.tsel_status_string(5) == "TSEL_ERR_DEVICE_CHECK"


def test_workspace_sizes_grow_with_the_problem(lib):
    import attention_score_vision_gb300 as tsel
    a = tsel.tsel_importance_workspace_size(1, 256, 256, 4)
    b = tsel.tsel_importance_workspace_size(30, 65536, 65536, 16)
    assert 1024 < a < b
    assert b % 256 == 0
    # padded LSE: H * 128 * (ceil(Tq/128) + G) floats at least
    assert b >= 16 * 128 * (512 + 30) * 4
    assert tsel.tsel_importance_workspace_size(-1, 1, 1, 1) == 0


def _call_importance(lib, **over):
    args = dict(q=16, qs=0, k=16, ks=0, cuq=16, cuk=16, G=1, tq=8, tk=8, mq=8, mk=8, H=4, Hkv=4,
                d=64, scale=0.0, flags=0, lse=0, scores=16, ws=256, wsb=1 << 20, stream=None)
    args.update(over)
    return lib.tsel_importance(args["q"], args["qs"], args["k"], args["ks"], args["cuq"], args["cuk"],
                               args["G"], args["tq"], args["tk"], args["mq"], args["mk"], args["H"],
                               args["Hkv"], args["d"], args["scale"], args["flags"], args["lse"] or None,
                               args["scores"], args["ws"], args["wsb"], args["stream"])


def test_importance_host_checks_fail_before_any_cuda_call(lib):
    # Fake (never dereferenced) addresses: every case below must be rejected
    # by the host checks, which run before anything touches the device.
    assert _call_importance(lib, d=72) == 2                 # unsupported head_dim
    assert _call_importance(lib, H=6, Hkv=4) == 1           # Hkv does not divide H
    assert _call_importance(lib, H=300, Hkv=300) == 1
    assert _call_importance(lib, q=8) == 1                  # misaligned q
    assert _call_importance(lib, qs=4 * 64 + 4) == 1        # row stride not 16-byte multiple
    assert _call_importance(lib, qs=64) == 1                # row stride < H*d
    assert _call_importance(lib, ws=128) == 3               # workspace misaligned
    assert _call_importance(lib, wsb=64) == 3               # workspace too small
    assert _call_importance(lib, cuq=0) == 1                # null cu_seqlens
    assert _call_importance(lib, flags=0x80) == 2           # unknown flag
    assert _call_importance(lib, flags=0x8 | 0x20) == 1     # fixed and moving reference
    assert _call_importance(lib, flags=0x2) == 1            # E4M3 inputs need softmax_scale
    assert _call_importance(lib, flags=0x2, scale=0.5, qs=4 * 64 + 4) == 1   # E4M3 row stride, 16-byte rule
    assert _call_importance(lib, flags=0x1, lse=0) == 1     # LSE-provided needs the lse input
    assert _call_importance(lib, tq=-1) == 1
    assert "head_dim=72" in (_call_importance(lib, d=72) and lib.tsel_last_error().decode())


def test_dynamic_budget_and_counted_gather_host_checks(lib):
    # permille arguments out of range, min > max, null pointers, workspace
    assert lib.tsel_dynamic_budget(16, 10, 16, 1, 1001, 0, 1000, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_dynamic_budget(16, 10, 16, 1, 500, 600, 500, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_dynamic_budget(16, 10, 16, 1, -1, 0, 1000, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_dynamic_budget(16, 10, None, 1, 500, 0, 1000, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_dynamic_budget(16, 10, 16, 1, 500, 0, 1000, None, 16, 256, 1024, None) == 1
    assert lib.tsel_dynamic_budget(16, 10, 16, 1, 500, 0, 1000, 16, 16, 128, 1024, None) == 3
    # counted gather needs the device count pointer
    assert lib.tsel_gather_compact_counted(16, 0, 8, 2, 16, 1, 16, 1, 4, 16, None, 2, 16, 16, 16,
                                           16, 256, 1024, None) == 1
    # top-B: only TSEL_KEEP_FROM_DEVICE (-1) is a valid negative total
    assert lib.tsel_select_topk(16, 10, 16, 1, 16, -2, 16, 16, 256, 1024, None) == 1


def test_topk_and_gather_host_checks(lib):
    assert lib.tsel_select_topk(16, 10, 16, 1, 16, 5, 16, 16, 128, 1024, None) == 3   # ws misaligned
    assert lib.tsel_select_topk(16, 10, None, 1, 16, 5, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_select_topk(16, -1, 16, 1, 16, 5, 16, 16, 256, 1024, None) == 1
    # gather: row bytes not a multiple of 16, bad elem size, pos_dim too large
    assert lib.tsel_gather_compact(16, 0, 7, 2, 16, 1, 16, 1, 4, 16, 2, 16, 16, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_gather_compact(16, 0, 8, 3, 16, 1, 16, 1, 4, 16, 2, 16, 16, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_gather_compact(16, 0, 8, 2, 16, 9, 16, 1, 4, 16, 2, 16, 16, 16, 16, 256, 1024, None) == 1
    assert lib.tsel_gather_compact(8, 0, 8, 2, 16, 1, 16, 1, 4, 16, 2, 16, 16, 16, 16, 256, 1024, None) == 1
